// Register-fragment building blocks of the stream-K mma.sync decode kernel
// behind the allocation-free entry (weights streamed per k-block, dequantised
// straight into mma.sync A fragments, x pre-permuted into B-fragment order in
// shared memory).
//
// Fragment mapping of one warp tile (32 output columns x one k-block of 64):
// thread (g = lane/4, t = lane%4) holds packed rows 2t and 2t+1 of the k-block
// for columns 4g..4g+3. Column 4g+2i+r is row g+8r of m16 tile i. For mma j
// (0..3), the thread's K slots (2t, 2t+1) are nibbles (j, j+4) of packed row
// 2t and slots (2t+8, 2t+9) the same nibbles of row 2t+1; x is permuted to the
// same K order when it is staged.
#pragma once

#include <cuda_fp16.h>

#include "kaio_device.cuh"

namespace kaio {
namespace {

template <int MT>
struct Frag {
  static constexpr int kRows = 8 * MT;        // padded batch rows
  static constexpr int kAcc = 8 * MT;         // f32 accumulators per thread
  static constexpr int kXkb = 128 * kRows;    // bytes of staged x per k-block
};

struct Ring {
  uint4 w0, w1;  // packed rows 2t and 2t+1, columns 4g .. 4g+3
  uint2 sc;      // scales of those 4 columns
};

__device__ __forceinline__ void load_ring(Ring& r, const uint32_t* __restrict__ w,
                                          const __half* __restrict__ s, int N, int kb, int col,
                                          int t, bool valid) {
  if (valid) {
    const uint32_t* p = w + static_cast<size_t>(kb * 8 + 2 * t) * N + col;
    r.w0 = ldg_stream_v4(p);
    r.w1 = ldg_stream_v4(p + N);
    r.sc = __ldg(reinterpret_cast<const uint2*>(s + static_cast<size_t>(kb >> 1) * N + col));
  } else {
    r.w0 = make_uint4(0, 0, 0, 0);
    r.w1 = r.w0;
    r.sc = make_uint2(0, 0);
  }
}

template <int MT>
__device__ __forceinline__ void compute_kb(float (&acc)[2][MT][4], const Ring& r,
                                           const unsigned char* xs_kb, int g, int t) {
  constexpr int R = Frag<MT>::kRows;
  uint4 xa[MT], xb[MT];
#pragma unroll
  for (int nt = 0; nt < MT; ++nt) {
    const unsigned char* base = xs_kb + (g + 8 * nt) * 64 + t * 16;
    xa[nt] = *reinterpret_cast<const uint4*>(base);
    xb[nt] = *reinterpret_cast<const uint4*>(base + 64 * R);
  }
  const uint32_t s2[4] = {
      __byte_perm(r.sc.x, 0, 0x1010), __byte_perm(r.sc.x, 0, 0x3232),
      __byte_perm(r.sc.y, 0, 0x1010), __byte_perm(r.sc.y, 0, 0x3232)};
  const PairedNibbles q0[4] = {PairedNibbles(r.w0.x), PairedNibbles(r.w0.y),
                               PairedNibbles(r.w0.z), PairedNibbles(r.w0.w)};
  const PairedNibbles q1[4] = {PairedNibbles(r.w1.x), PairedNibbles(r.w1.y),
                               PairedNibbles(r.w1.z), PairedNibbles(r.w1.w)};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t b0[MT], b1[MT];
#pragma unroll
    for (int nt = 0; nt < MT; ++nt) {
      b0[nt] = (j == 0) ? xa[nt].x : (j == 1) ? xa[nt].y : (j == 2) ? xa[nt].z : xa[nt].w;
      b1[nt] = (j == 0) ? xb[nt].x : (j == 1) ? xb[nt].y : (j == 2) ? xb[nt].z : xb[nt].w;
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint32_t a[4] = {q0[2 * i].pair(j, s2[2 * i]), q0[2 * i + 1].pair(j, s2[2 * i + 1]),
                             q1[2 * i].pair(j, s2[2 * i]), q1[2 * i + 1].pair(j, s2[2 * i + 1])};
#pragma unroll
      for (int nt = 0; nt < MT; ++nt) mma_16816(acc[i][nt], a, b0[nt], b1[nt]);
    }
  }
}

// Stage x[0:8*MT, kb0 .. kb0+nkb) into shared memory in B-fragment order.
// Per k-block the layout is [h][m][t] pieces of 16 bytes; piece (h, m, t) holds
// x[m, 64kb + 16t + 8h .. +7] regrouped as pairs (e0,e4) (e1,e5) (e2,e6) (e3,e7).
// Rows m >= M are zero.
template <int MT>
__device__ __forceinline__ void stage_x(unsigned char* xs, const __half* __restrict__ x, int M,
                                        int K, int kb0, int nkb, int tid, int nthreads) {
  constexpr int R = Frag<MT>::kRows;
  const int pieces = nkb * 8 * R;
  for (int pc = tid; pc < pieces; pc += nthreads) {
    const int kbl = pc / (8 * R);
    const int rem = pc % (8 * R);
    const int h = rem / (4 * R);
    const int m = (rem % (4 * R)) >> 2;
    const int tt = rem & 3;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (m < M)
      v = __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(m) * K + (kb0 + kbl) * 64 +
                                               16 * tt + 8 * h));
    uint4 o;
    o.x = __byte_perm(v.x, v.z, 0x5410);
    o.y = __byte_perm(v.x, v.z, 0x7632);
    o.z = __byte_perm(v.y, v.w, 0x5410);
    o.w = __byte_perm(v.y, v.w, 0x7632);
    *reinterpret_cast<uint4*>(xs + static_cast<size_t>(pc) * 16) = o;
  }
}

}  // namespace
}  // namespace kaio
