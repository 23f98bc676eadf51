// W4A16 fused QKV projection, decode-sized M (1..16), split over K across the
// CTAs of a thread-block cluster.
//
// What it computes ("kaio-candle -- src/qkv_project_int4.rs", doc comment of
// qkv_project_int4): out_p[m, n] = f16(sum_k x[m, k] * RN_f16(int4(W_p[k, n]) *
// s_p[k/128, n])), f32 accumulation, f32 -> f16 in-kernel.
//
// Design (one GPU, sm_103a). A column group (256 output columns of one
// projection) is owned by one cluster of S CTAs; CTA rank r covers a
// contiguous range of 128-row K groups (one scale row each).
// * A producer warp issues TMA copies for the CTA's packed weights (one 2 KB
//   128B-swizzled box of 16 packed rows x 32 columns per column warp and K group)
//   into a ring of 16 KB stages sized to hold as much of the CTA's share as
//   shared memory allows -- for decode shapes usually all of it, so every byte
//   the CTA needs is requested in the first microsecond -- plus one copy of
//   the scale rows of its range.
// * 16 consumer warps (8 column warps x 2 k-warps) stage x once in B-fragment
//   order, then per K group read their packed words from the swizzled box
//   (conflict-free), dequantise in registers into mma.sync A fragments and
//   accumulate over K on the tensor cores (see decode_frag.cuh).
// * Reduction: k-warps through shared memory, then the S CTAs of the cluster
//   through distributed shared memory: each rank finishes some column warps by
//   reading the S partials in rank order (deterministic) and writes f16.
// No global scratch, no atomics. Every mbarrier wait is bounded; both cluster
// barriers are always reached by every thread, so a timed-out wait cannot
// leave a peer CTA blocked.
#include <cuda.h>
#include <cuda_fp16.h>

#include <map>
#include <mutex>
#include <utility>

#include "decode_frag.cuh"
#include "kaio_device.cuh"
#include "kaio_internal.h"

namespace kaio {

__device__ unsigned g_dc_err = 0;

namespace {

constexpr int kCW = 8;                      // column warps (32 columns each)
constexpr int kKW = 2;                      // k-warps: k-block 0 / 1 of each K group
constexpr int kConsumers = kCW * kKW;       // 16 warps
constexpr int kThreads = (kConsumers + 1) * 32;  // + producer warp = 544
constexpr int kGroupCols = kCW * 32;        // 256
constexpr int kStageBytes = 16384;          // one K group (16 packed rows) x 256 columns
constexpr int kBoxBytes = 2048;             // 16 packed rows x 32 columns (128 B rows)
constexpr int kMaxStages = 16;
constexpr int kScaleRowBytes = kGroupCols * 2;

struct ClusterParams {
  const __half* x;
  __half* out[3];
  int M, N, K;
  int groups_per_proj;   // ceil(N / 256)
  int S;                 // cluster size = number of K ranges per column group
  int ng;                // K / 128
  int nst;               // ring stages
  int sbox;              // scale rows per TMA box
  int x_off, s_off;      // shared-memory offsets of staged x and scales
};

template <int MT>
__global__ void __launch_bounds__(kThreads, 1)
    decode_cluster_kernel(const __grid_constant__ CUtensorMap tw0, const __grid_constant__ CUtensorMap tw1,
                          const __grid_constant__ CUtensorMap tw2, const __grid_constant__ CUtensorMap ts0,
                          const __grid_constant__ CUtensorMap ts1, const __grid_constant__ CUtensorMap ts2,
                          const ClusterParams p) {
  constexpr int XKB = Frag<MT>::kXkb;
  constexpr int F = Frag<MT>::kAcc;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = align_smem_1024(smem_raw);
  __shared__ __align__(8) uint64_t full[kMaxStages], empty[kMaxStages], sbar;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_ctarank());
  const int gi = blockIdx.x / p.S;
  const int proj = gi / p.groups_per_proj;
  const int col0 = (gi % p.groups_per_proj) * kGroupCols;
  const int g_begin = rank * p.ng / p.S;
  const int nsg = (rank + 1) * p.ng / p.S - g_begin;   // K groups (= ring stages) of this CTA
  volatile int* abort = &abort_flag;

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.nst; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumers);
    }
    mbar_init(&sbar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumers) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const CUtensorMap* tw = proj == 0 ? &tw0 : (proj == 1 ? &tw1 : &tw2);
      const CUtensorMap* ts = proj == 0 ? &ts0 : (proj == 1 ? &ts1 : &ts2);
      tma_prefetch_desc(tw);
      tma_prefetch_desc(ts);
      const int nsbox = (nsg + p.sbox - 1) / p.sbox;
      mbar_arrive_expect_tx(&sbar, static_cast<uint32_t>(nsbox * p.sbox * kScaleRowBytes));
      for (int b = 0; b < nsbox; ++b)
        tma_load_2d(smem + p.s_off + b * p.sbox * kScaleRowBytes, ts, &sbar, col0, g_begin + b * p.sbox);
      uint32_t fills[kMaxStages];
      for (int i = 0; i < kMaxStages; ++i) fills[i] = 0;
      for (int i = 0; i < nsg; ++i) {
        const int slot = i % p.nst;
        if (i >= p.nst && !mbar_wait(&empty[slot], ((i / p.nst) - 1) & 1, abort, &g_dc_err)) break;
        ++fills[slot];
        mbar_arrive_expect_tx(&full[slot], kStageBytes);
        unsigned char* dst = smem + slot * kStageBytes;
        const int row = (g_begin + i) * 16;
#pragma unroll
        for (int cw = 0; cw < kCW; ++cw)
          tma_load_2d(dst + cw * kBoxBytes, tw, &full[slot], col0 + 32 * cw, row);
      }
      // No copy may still be landing when the CTA moves on or exits.
      for (int s2 = 0; s2 < p.nst; ++s2)
        if (fills[s2]) mbar_wait_drain(&full[s2], (fills[s2] - 1) & 1, &g_dc_err);
      mbar_wait_drain(&sbar, 0, &g_dc_err);
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int cw = warp % kCW, kw = warp / kCW;
    const int g = lane >> 2, t = lane & 3;
    stage_x<MT>(smem + p.x_off, p.x, p.M, p.K, g_begin * 2, nsg * 2, threadIdx.x, kConsumers * 32);
    named_sync(1, kConsumers * 32);

    float acc[2][MT][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int nt = 0; nt < MT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[i][nt][e] = 0.f;

    if (mbar_wait(&sbar, 0, abort, &g_dc_err)) {
      const int r0 = 8 * kw + 2 * t, r1 = r0 + 1;
      const int o0 = r0 * 128 + ((g ^ (r0 & 7)) << 4);
      const int o1 = r1 * 128 + ((g ^ (r1 & 7)) << 4);
      const unsigned char* sc = smem + p.s_off + (cw * 32 + 4 * g) * 2;
      for (int i = 0; i < nsg; ++i) {
        const int slot = i % p.nst;
        if (!mbar_wait(&full[slot], (i / p.nst) & 1, abort, &g_dc_err)) break;
        const unsigned char* box = smem + slot * kStageBytes + cw * kBoxBytes;
        Ring r;
        r.w0 = *reinterpret_cast<const uint4*>(box + o0);
        r.w1 = *reinterpret_cast<const uint4*>(box + o1);
        r.sc = *reinterpret_cast<const uint2*>(sc + i * kScaleRowBytes);
        compute_kb<MT>(acc, r, smem + p.x_off + static_cast<size_t>(2 * i + kw) * XKB, g, t);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
      }
    }

    // k-warp reduction; the ring is free once every consumer is past its loop.
    float f[F];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int nt = 0; nt < MT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) f[(i * MT + nt) * 4 + e] = acc[i][nt][e];
    float* red_kw = reinterpret_cast<float*>(smem);                 // [kCW][32][F]
    float* red_cl = red_kw + kCW * 32 * F;                          // [kCW][32][F]
    named_sync(1, kConsumers * 32);
    if (kw == 1) {
#pragma unroll
      for (int q = 0; q < F; q += 4)
        *reinterpret_cast<float4*>(red_kw + (cw * 32 + lane) * F + q) =
            make_float4(f[q], f[q + 1], f[q + 2], f[q + 3]);
    }
    named_sync(1, kConsumers * 32);
    if (kw == 0) {
#pragma unroll
      for (int q = 0; q < F; q += 4) {
        const float4 o = *reinterpret_cast<const float4*>(red_kw + (cw * 32 + lane) * F + q);
        *reinterpret_cast<float4*>(red_cl + (cw * 32 + lane) * F + q) =
            make_float4(f[q] + o.x, f[q + 1] + o.y, f[q + 2] + o.z, f[q + 3] + o.w);
      }
    }
  }

  // Cluster reduction: rank r finishes the column warps cw with cw % S == r.
  __syncwarp();
  cluster_sync_all();
  if (warp < kCW && warp % p.S == rank) {
    const int cw = warp;
    const int g = lane >> 2, t = lane & 3;
    float f[F];
#pragma unroll
    for (int q = 0; q < F; ++q) f[q] = 0.f;
    const uint32_t local = smem_u32(smem) + static_cast<uint32_t>((kCW * 32 * F + (cw * 32 + lane) * F) * 4);
    for (int r = 0; r < p.S; ++r) {
      const uint32_t remote = dsmem_map(local, static_cast<uint32_t>(r));
#pragma unroll
      for (int q = 0; q < F; q += 4) {
        const float4 o = dsmem_ld_f4(remote + q * 4);
        f[q] += o.x; f[q + 1] += o.y; f[q + 2] += o.z; f[q + 3] += o.w;
      }
    }
    const int col = col0 + cw * 32 + 4 * g;
    if (col < p.N) {
      __half* out = proj == 0 ? p.out[0] : (proj == 1 ? p.out[1] : p.out[2]);
#pragma unroll
      for (int nt = 0; nt < MT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int m = 8 * nt + 2 * t + e;
          if (m < p.M) {
            const __half2 lo = __floats2half2_rn(f[(0 * MT + nt) * 4 + e], f[(0 * MT + nt) * 4 + 2 + e]);
            const __half2 hi = __floats2half2_rn(f[(1 * MT + nt) * 4 + e], f[(1 * MT + nt) * 4 + 2 + e]);
            uint2 v;
            v.x = *reinterpret_cast<const uint32_t*>(&lo);
            v.y = *reinterpret_cast<const uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(out + static_cast<size_t>(m) * p.N + col) = v;
          }
        }
    }
  }
  __syncwarp();
  cluster_sync_all();   // peers keep their partials until every reader is done
}

// Dynamic shared memory: the kernel's limit is raised to kSmemAttr; layouts use
// at most kSmemMax of it (1 KB is kept for aligning the base to 1024 bytes).
constexpr int kSmemAttr = 232448 - 1024;  // opt-in per-block limit minus static shared memory
constexpr int kSmemMax = kSmemAttr - 1024;

int max_active_clusters(int mt, int S, int dev) {
  static std::mutex mu;
  static std::map<std::pair<int, int>, int> cache;   // (dev, mt*16 + S) -> clusters
  std::lock_guard<std::mutex> lk(mu);
  const auto key = std::make_pair(dev, mt * 16 + S);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  const void* kern = mt == 1 ? reinterpret_cast<const void*>(decode_cluster_kernel<1>)
                             : reinterpret_cast<const void*>(decode_cluster_kernel<2>);
  int n = 0;
  if (ensure_smem_limit(kern, kSmemAttr) == cudaSuccess) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(S * 64));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemAttr;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(S);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
  }
  cache[key] = n;
  return n;
}

}  // namespace

ClusterPlan plan_decode_cluster(int M, int N, int K, int num_sms, int dev) {
  ClusterPlan pl{};
  pl.mt = (M <= 8) ? 1 : 2;
  pl.groups_per_proj = (N + kGroupCols - 1) / kGroupCols;
  pl.groups = 3 * pl.groups_per_proj;
  pl.ng = K / 128;
  const int xkb = 1024 * pl.mt;
  long long best = -1;
  for (int S = 1; S <= 8 && S <= pl.ng; ++S) {
    const int range = (pl.ng + S - 1) / S;
    const int sbox = std::min(8, pl.ng);
    const int sbytes = ((range + sbox - 1) / sbox) * sbox * kScaleRowBytes;
    const int xbytes = range * 2 * xkb;
    const int fixed = xbytes + sbytes;
    if (fixed + 2 * kStageBytes > kSmemMax) continue;
    const int slots = max_active_clusters(pl.mt, S, dev);
    if (slots <= 0) continue;
    const long long waves = (pl.groups + slots - 1) / slots;
    const long long est = waves * range;
    if (best < 0 || est < best) {
      best = est;
      pl.S = S;
      pl.sbox = sbox;
      pl.nst = std::min(std::min(range, kMaxStages), (kSmemMax - fixed) / kStageBytes);
      pl.nst = std::max(pl.nst, 2);
      pl.s_off = pl.nst * kStageBytes;
      pl.x_off = pl.s_off + sbytes;
      pl.smem = static_cast<size_t>(pl.x_off + xbytes) + 1024;
      pl.est_groups = est;
    }
  }
  // The k-warp and cluster partials reuse the ring: it must hold 2 x 8 x 32 x 8*mt floats.
  pl.ok = best > 0 && pl.nst * kStageBytes >= 2 * kCW * 32 * 8 * pl.mt * 4;
  return pl;
}

cudaError_t launch_decode_cluster(const __half* x, const uint32_t* const w[3],
                                  const __half* const s[3], __half* const out[3], int M, int N, int K,
                                  const ClusterPlan& pl, cudaStream_t stream) {
  CUtensorMap tw[3], ts[3];
  for (int q = 0; q < 3; ++q) {
    CUresult r = encode_tensor_map_2d(&tw[q], CU_TENSOR_MAP_DATA_TYPE_UINT32, w[q], N, K / 8,
                                      static_cast<uint64_t>(N) * 4, 32, 16, CU_TENSOR_MAP_SWIZZLE_128B);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    r = encode_tensor_map_2d(&ts[q], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, s[q], N, K / 128,
                             static_cast<uint64_t>(N) * 2, kGroupCols, pl.sbox, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  ClusterParams p{};
  p.x = x;
  for (int q = 0; q < 3; ++q) p.out[q] = out[q];
  p.M = M;
  p.N = N;
  p.K = K;
  p.groups_per_proj = pl.groups_per_proj;
  p.S = pl.S;
  p.ng = pl.ng;
  p.nst = pl.nst;
  p.sbox = pl.sbox;
  p.x_off = pl.x_off;
  p.s_off = pl.s_off;
  const void* kern = pl.mt == 1 ? reinterpret_cast<const void*>(decode_cluster_kernel<1>)
                                : reinterpret_cast<const void*>(decode_cluster_kernel<2>);
  cudaError_t e = ensure_smem_limit(kern, kSmemAttr);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(pl.groups * pl.S));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(pl.S);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (pl.mt == 1)
    e = cudaLaunchKernelEx(&cfg, decode_cluster_kernel<1>, tw[0], tw[1], tw[2], ts[0], ts[1], ts[2], p);
  else
    e = cudaLaunchKernelEx(&cfg, decode_cluster_kernel<2>, tw[0], tw[1], tw[2], ts[0], ts[1], ts[2], p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

unsigned read_and_clear_decode_errors() {
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_dc_err, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
  const unsigned zero = 0;
  cudaMemcpyToSymbol(g_dc_err, &zero, sizeof(zero));
  return v;
}

}  // namespace kaio
