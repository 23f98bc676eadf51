// W4A16 fused QKV projection, decode-sized M (1..16): a weight-streaming
// kernel bound by the packed-weight bytes.
//
// What it computes ("kaio-candle -- src/qkv_project_int4.rs", doc comment of
// qkv_project_int4): for p in {Q, K, V},
//     out_p[m, n] = f16( sum_k x[m, k] * RN_f16(int4(W_p[k, n]) * s_p[k/128, n]) )
// with f32 accumulation and the f32 -> f16 cast done here.
//
// Design (one GPU, sm_103a):
// * Work is the set of units (column group, k-block): a column group is 256
//   output columns of one projection (8 warp tiles of 32 columns), a k-block is
//   64 K-rows (8 packed rows). The units are laid out group-major and cut into
//   one contiguous, equal share per CTA (stream-K), one CTA per SM, so every SM
//   streams the same number of weight bytes whatever the shape.
// * A CTA has 16 warps: 8 column warps x 2 k-warps. Each warp streams its
//   packed weights straight from HBM into registers with 128-bit
//   L1-bypassing loads, several k-blocks ahead, and never stages them in
//   shared memory.
// * The activations of the CTA's k-range are staged once in shared memory,
//   already permuted into mma.sync B-fragment order, and shared by all 8
//   column tiles.
// * Dequantisation happens in registers and yields mma.sync A fragments
//   directly. The reduction over K runs on the tensor cores
//   (m16n8k16, f32 accumulate): output columns are the MMA's M side and the
//   batch rows its N side. Within one MMA the K order is free as long as A
//   and B agree, so each thread's fragment takes nibble pairs (j, j+4) of a
//   packed word as they fall out of the mask trick, and x is permuted to match.
// * k-warps are reduced through shared memory. A group split across CTAs is
//   finished by the last CTA to arrive (per-group counter); it sums the
//   partials in CTA order, so the result is deterministic, then resets the
//   counter for the next launch.
#include <cuda_fp16.h>

#include <mutex>

#include "decode_frag.cuh"
#include "kaio_device.cuh"
#include "kaio_internal.h"

namespace kaio {
namespace {

constexpr int kCW = 8;                 // column warps per CTA
constexpr int kKW = 2;                 // k-warps per column tile
constexpr int kWarps = kCW * kKW;      // 16
constexpr int kThreads = kWarps * 32;  // 512
constexpr int kGroupCols = kCW * 32;   // 256 output columns per group
constexpr int kDepth = 4;              // k-blocks of weights in flight per warp

// Unit range of CTA c: [c*U/G, (c+1)*U/G).
__device__ __forceinline__ long long unit_begin(long long c, long long U, long long G) {
  return (c * U) / G;
}
// The CTA whose range contains unit u.
__device__ __forceinline__ long long cta_of_unit(long long u, long long U, long long G) {
  return ((u + 1) * G - 1) / U;
}

template <int MT>
__global__ void __launch_bounds__(kThreads, 1) decode_w4a16_kernel(const DecodeParams p) {
  constexpr int R = Frag<MT>::kRows;
  constexpr int XKB = Frag<MT>::kXkb;
  constexpr int F = Frag<MT>::kAcc;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* xs = smem;                                                   // staged x
  float* red = reinterpret_cast<float*>(smem + static_cast<size_t>(p.xmax_kb) * XKB);  // [kCW][32][F]
  __shared__ int s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cw = warp % kCW, kw = warp / kCW;
  const int g = lane >> 2, t = lane & 3;
  const long long U = p.units, G = p.ctas, c = blockIdx.x;
  const long long ub = unit_begin(c, U, G), ue = unit_begin(c + 1, U, G);

  for (long long u = ub; u < ue;) {
    const int gi = static_cast<int>(u / p.nkb);
    const int kb0 = static_cast<int>(u % p.nkb);
    const long long seg_end = kb0 + (ue - u);
    const int kb1 = seg_end < p.nkb ? static_cast<int>(seg_end) : p.nkb;
    const int proj = gi / p.groups_per_proj;
    const int gc = gi % p.groups_per_proj;
    const int col = gc * kGroupCols + cw * 32 + 4 * g;   // first of this thread's 4 columns
    const bool col_ok = col < p.N;
    const uint32_t* __restrict__ w = p.w[proj];
    const __half* __restrict__ s = p.s[proj];

    float acc[2][MT][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int nt = 0; nt < MT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[i][nt][e] = 0.f;

    for (int ck0 = kb0; ck0 < kb1; ck0 += p.xmax_kb) {
      const int ck1 = min(kb1, ck0 + p.xmax_kb);
      const int nk = (ck1 - ck0 - kw + kKW - 1) / kKW;   // this warp's k-blocks in the chunk
      Ring ring[kDepth];
#pragma unroll
      for (int d = 0; d < kDepth; ++d)
        if (d < nk) load_ring(ring[d], w, s, p.N, ck0 + kw + kKW * d, col, t, col_ok);

      // Stage x[0:R, chunk] permuted into B-fragment order. Piece layout per
      // k-block: [h][m][t] of 16 bytes; piece (h, m, t) holds the 8 K-values at
      // 16t + 8h .. +7 regrouped as pairs (e0,e4) (e1,e5) (e2,e6) (e3,e7).
      const int pieces = (ck1 - ck0) * 8 * R;
      for (int pc = threadIdx.x; pc < pieces; pc += kThreads) {
        const int kbl = pc / (8 * R);
        const int rem = pc % (8 * R);
        const int h = rem / (4 * R);
        const int m = (rem % (4 * R)) >> 2;
        const int tt = rem & 3;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (m < p.M)
          v = __ldg(reinterpret_cast<const uint4*>(
              p.x + static_cast<size_t>(m) * p.K + (ck0 + kbl) * 64 + 16 * tt + 8 * h));
        uint4 o;
        o.x = __byte_perm(v.x, v.z, 0x5410);
        o.y = __byte_perm(v.x, v.z, 0x7632);
        o.z = __byte_perm(v.y, v.w, 0x5410);
        o.w = __byte_perm(v.y, v.w, 0x7632);
        *reinterpret_cast<uint4*>(xs + static_cast<size_t>(pc) * 16) = o;
      }
      __syncthreads();

      for (int base = 0; base < nk; base += kDepth) {
#pragma unroll
        for (int d = 0; d < kDepth; ++d) {
          const int i = base + d;
          if (i < nk) {
            const int kbl = kw + kKW * i;
            compute_kb<MT>(acc, ring[d], xs + static_cast<size_t>(kbl) * XKB, g, t);
            if (i + kDepth < nk)
              load_ring(ring[d], w, s, p.N, ck0 + kw + kKW * (i + kDepth), col, t, col_ok);
          }
        }
      }
      __syncthreads();  // x chunk fully consumed
    }

    // Reduce the k-warps: kw = 1 publishes, kw = 0 accumulates.
    float f[F];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int nt = 0; nt < MT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) f[(i * MT + nt) * 4 + e] = acc[i][nt][e];
    float* my_red = red + (cw * 32 + lane) * F;
    if (kw == 1) {
#pragma unroll
      for (int q = 0; q < F; q += 4)
        *reinterpret_cast<float4*>(my_red + q) = make_float4(f[q], f[q + 1], f[q + 2], f[q + 3]);
    }
    __syncthreads();
    if (kw == 0) {
#pragma unroll
      for (int q = 0; q < F; q += 4) {
        const float4 o = *reinterpret_cast<const float4*>(my_red + q);
        f[q] += o.x; f[q + 1] += o.y; f[q + 2] += o.z; f[q + 3] += o.w;
      }
    }

    const bool full = (kb0 == 0 && kb1 == p.nkb);
    bool finish = full;
    if (!full) {
      // Partial: publish to this CTA's slot (0 = first segment, 1 = last).
      const int si = (u == ub) ? 0 : 1;
      if (kw == 0) {
        float* slot = p.partials + ((static_cast<size_t>(c) * 2 + si) * kCW + cw) * 32 * F + lane * F;
#pragma unroll
        for (int q = 0; q < F; q += 4)
          __stcg(reinterpret_cast<float4*>(slot + q), make_float4(f[q], f[q + 1], f[q + 2], f[q + 3]));
        __threadfence();
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        const unsigned add = static_cast<unsigned>(kb1 - kb0);
        const unsigned prev = atomicAdd(p.counters + gi, add);
        s_last = (prev + add == static_cast<unsigned>(p.nkb)) ? 1 : 0;
      }
      __syncthreads();
      finish = s_last != 0;
      if (finish && kw == 0) {
        __threadfence();
        // Sum every contributor's partial in CTA order.
        const long long gu0 = static_cast<long long>(gi) * p.nkb;
        const long long c0 = cta_of_unit(gu0, U, G);
        const long long c1 = cta_of_unit(gu0 + p.nkb - 1, U, G);
#pragma unroll
        for (int q = 0; q < F; ++q) f[q] = 0.f;
        for (long long cc = c0; cc <= c1; ++cc) {
          const long long cb = unit_begin(cc, U, G);
          const int si2 = (cb / p.nkb == gi) ? 0 : 1;
          const float* slot =
              p.partials + ((static_cast<size_t>(cc) * 2 + si2) * kCW + cw) * 32 * F + lane * F;
#pragma unroll
          for (int q = 0; q < F; q += 4) {
            const float4 o = __ldcg(reinterpret_cast<const float4*>(slot + q));
            f[q] += o.x; f[q + 1] += o.y; f[q + 2] += o.z; f[q + 3] += o.w;
          }
        }
        if (threadIdx.x == 0) p.counters[gi] = 0;  // ready for the next launch
      }
    }

    if (finish && kw == 0 && col_ok) {
      __half* out = p.out[proj];
#pragma unroll
      for (int nt = 0; nt < MT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int m = 8 * nt + 2 * t + e;
          if (m < p.M) {
            // columns col+0..3 = (i=0,r=0) (i=0,r=1) (i=1,r=0) (i=1,r=1)
            const __half2 lo = __floats2half2_rn(f[(0 * MT + nt) * 4 + e], f[(0 * MT + nt) * 4 + 2 + e]);
            const __half2 hi = __floats2half2_rn(f[(1 * MT + nt) * 4 + e], f[(1 * MT + nt) * 4 + 2 + e]);
            uint2 v;
            v.x = *reinterpret_cast<const uint32_t*>(&lo);
            v.y = *reinterpret_cast<const uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(out + static_cast<size_t>(m) * p.N + col) = v;
          }
        }
    }
    __syncthreads();  // the reduction buffer and s_last are reused by the next segment
    u += kb1 - kb0;
  }
}

}  // namespace

size_t decode_smem_bytes(int mt, int xmax_kb) {
  const int rows = 8 * mt;
  return static_cast<size_t>(xmax_kb) * 128 * rows + static_cast<size_t>(kCW) * 32 * 8 * mt * 4;
}

DecodePlan plan_decode(int M, int N, int K, int num_sms) {
  DecodePlan pl{};
  pl.mt = (M <= 8) ? 1 : 2;
  pl.groups_per_proj = (N + kGroupCols - 1) / kGroupCols;
  pl.nkb = K / 64;
  pl.units = 3LL * pl.groups_per_proj * pl.nkb;
  pl.ctas = static_cast<int>(std::min<long long>(pl.units, num_sms));
  const long long per_cta = (pl.units + pl.ctas - 1) / pl.ctas;
  // x staged per chunk: at most ~192 KB of shared memory (one CTA per SM).
  const int cap = (pl.mt == 1) ? 192 : 96;
  pl.xmax_kb = static_cast<int>(std::min<long long>(std::min<long long>(per_cta, pl.nkb), cap));
  pl.smem = decode_smem_bytes(pl.mt, pl.xmax_kb);
  pl.partial_floats = static_cast<size_t>(pl.ctas) * 2 * kCW * 32 * 8 * pl.mt;
  pl.counters = 3 * pl.groups_per_proj;
  return pl;
}

// ---------------------------------------------------------------------------
// Allocation-free variant of the decode launch.
//
// Some callers cannot allocate device memory: code that runs inside another
// runtime's memory budget (inference engines and plugin hosts that hand out
// every byte themselves and forbid cudaMalloc), processes whose device memory
// is fully reserved up front, and real-time paths where an allocation's
// implicit synchronisation or failure is not acceptable. For them this
// stream-K decode kernel, whose split-K needs global scratch (per-group
// arrival counters and the partial sums), keeps that scratch in this fixed
// array and allocates nothing. Every GPU that loads the library holds
// these bytes until the process exits. All calls share the one array: calls
// whose kernels overlap on the GPU (different streams, no ordering between
// them) race on it and give wrong results; order them on one stream.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
constexpr size_t kNoAllocCounterBytes = 64u << 10;                  // 16384 group counters
static_assert(kNoAllocScratchBytes > kNoAllocCounterBytes, "scratch layout");

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
unsigned char* g_noalloc_ptr[kMaxDevices] = {};
}  // namespace

// Device address of the scratch array on the current device. The array's name
// in host code is only a host-side stand-in, so the address is looked up once
// per device (this first call should come before any stream capture).
static cudaError_t noalloc_scratch(int dev, unsigned char** out) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = static_cast<unsigned char*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

int noalloc_max_counters() { return static_cast<int>(kNoAllocCounterBytes / sizeof(unsigned)); }

cudaError_t launch_decode_noalloc(DecodeParams prm, int dev, int num_sms, cudaStream_t stream) {
  unsigned char* base = nullptr;
  cudaError_t e = noalloc_scratch(dev, &base);
  if (e != cudaSuccess) return e;
  // As many CTAs as the partial-sum region holds (all SMs on a GB300).
  const int mt = (prm.M <= 8) ? 1 : 2;
  const size_t per_cta = static_cast<size_t>(2) * kCW * 32 * 8 * mt * sizeof(float);
  const int fit = static_cast<int>((kNoAllocScratchBytes - kNoAllocCounterBytes) / per_cta);
  const DecodePlan pl = plan_decode(prm.M, prm.N, prm.K, std::min(num_sms, fit));
  if (static_cast<size_t>(pl.counters) * sizeof(unsigned) > kNoAllocCounterBytes)
    return cudaErrorInvalidValue;
  prm.groups_per_proj = pl.groups_per_proj;
  prm.nkb = pl.nkb;
  prm.units = pl.units;
  prm.ctas = pl.ctas;
  prm.xmax_kb = pl.xmax_kb;
  prm.counters = reinterpret_cast<unsigned*>(base);
  prm.partials = reinterpret_cast<float*>(base + kNoAllocCounterBytes);
  // The counters must start at zero; the array keeps whatever the last call left.
  e = cudaMemsetAsync(prm.counters, 0, static_cast<size_t>(pl.counters) * sizeof(unsigned), stream);
  if (e != cudaSuccess) return e;
  const void* kern = (pl.mt == 1) ? reinterpret_cast<const void*>(decode_w4a16_kernel<1>)
                                   : reinterpret_cast<const void*>(decode_w4a16_kernel<2>);
  // Raise (never lower) the kernel's dynamic shared-memory limit.
  cudaFuncAttributes fa{};
  e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (static_cast<size_t>(fa.maxDynamicSharedSizeBytes) < pl.smem) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(pl.smem));
    if (e != cudaSuccess) return e;
  }
  if (pl.mt == 1)
    decode_w4a16_kernel<1><<<pl.ctas, kThreads, pl.smem, stream>>>(prm);
  else
    decode_w4a16_kernel<2><<<pl.ctas, kThreads, pl.smem, stream>>>(prm);
  return cudaGetLastError();
}

}  // namespace kaio
