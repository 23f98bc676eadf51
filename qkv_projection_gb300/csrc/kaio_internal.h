// Internal (non-exported) declarations shared by the translation units of
// libkaio_qkv: kernel parameter blocks, launch plans and launchers.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstddef>
#include <cstdint>

namespace kaio {

// ---------------------------------------------------------------- decode path
struct DecodeParams {
  const __half* x;          // [M, K]
  const uint32_t* w[3];     // [K/8, N] each
  const __half* s[3];       // [K/128, N] each
  __half* out[3];           // [M, N] each
  int M, N, K;
  int groups_per_proj;      // ceil(N / 256)
  int nkb;                  // K / 64
  long long units;          // 3 * groups_per_proj * nkb
  int ctas;                 // grid size
  int xmax_kb;              // k-blocks of x staged in shared memory at once
  float* partials;          // [ctas][2][8][32][8*mt] split-K partial sums
  unsigned* counters;       // [3 * groups_per_proj], zero between launches
};

struct DecodePlan {
  int mt;                   // 1: M <= 8, 2: M <= 16
  int groups_per_proj;
  int nkb;
  long long units;
  int ctas;
  int xmax_kb;
  size_t smem;
  size_t partial_floats;
  int counters;
};

// Stream-K mma.sync decode kernel, run only by the allocation-free entry point.
DecodePlan plan_decode(int M, int N, int K, int num_sms);

// Allocation-free decode launch: split-K scratch in a fixed device array of
// kNoAllocScratchBytes (the first 64 KiB hold group counters). `prm` needs only
// the tensors and M, N, K; the plan and scratch pointers are filled in here.
constexpr size_t kNoAllocScratchBytes = 8u << 20;
int noalloc_max_counters();
cudaError_t launch_decode_noalloc(DecodeParams prm, int dev, int num_sms, cudaStream_t stream);

// tcgen05 decode (M <= 16): 128-column tiles over the three projections, split
// over K across a cluster of S CTAs.
struct TcDecodePlan {
  bool ok;
  int tiles;   // ceil(N / 128)
  int ng;      // K / 128
  int S;       // cluster size
};
TcDecodePlan plan_tc_decode(int M, int N, int K, int dev);
cudaError_t launch_tc_decode(const __half* x, const uint32_t* const w[3], const __half* const s[3],
                             __half* const out[3], int M, int N, int K, const TcDecodePlan& pl,
                             cudaStream_t stream);
// The INT4 decode kernel with every pipeline wait limited to wait_ns (a test
// of the bounded-wait timeout path; the regular launch uses 2 s).
cudaError_t launch_tc_decode_wait_limit(const __half* x, const uint32_t* const w[3], const __half* const s[3],
                                        __half* const out[3], int M, int N, int K, const TcDecodePlan& pl,
                                        unsigned long long wait_ns, cudaStream_t stream);
// The same kernel for INT8 weights u32[K/4, N] (byte i = K-row 4r+i) with
// one f32 scale per projection.
TcDecodePlan plan_tc_decode_int8(int M, int N, int K, int dev);
cudaError_t launch_tc_decode_int8(const __half* x, const uint32_t* const w[3], const float scale[3],
                                  __half* const out[3], int M, int N, int K, const TcDecodePlan& pl,
                                  cudaStream_t stream);
unsigned read_and_clear_tc_decode_errors();

// ------------------------------------------------- per-group dequantisation
enum class FloatType { F32, F64, F16, BF16 };
// dx[i, j] = dy[i, j] * scale[i, j / group] over [outer, axis], in type t.
cudaError_t launch_dequant_group_backward(FloatType t, const void* dy, const void* scale, void* dx,
                                          int outer, int axis, int group, int num_sms, cudaStream_t stream);
// out[i, j] = t(q[i, j]) * scale[i, j / group], q int8 (or uint8 if q_unsigned).
cudaError_t launch_dequant_group_forward(FloatType t, bool q_unsigned, const void* q, const void* scale,
                                         void* out, int outer, int axis, int group, int num_sms,
                                         cudaStream_t stream);

// ------------------------------------------------- tensor-core (tcgen05) paths
struct GemmShape {
  int M, N, K;              // C[M, N] = sum_k Aop[M, k] * Bop[k, N]
};

// Dense f16 x f16 -> f32 accumulate, stored as f32 or (c_f16) f16. a_mn / b_mn
// select the operand storage:
//   Aop K-major: A stored [M][K];  MN-major: A stored [K][M]
//   Bop K-major: B stored [N][K];  MN-major: B stored [K][N]
cudaError_t launch_tc_gemm(const void* a, const void* b, void* c, GemmShape sh, bool a_mn,
                           bool b_mn, bool c_f16, int num_sms, cudaStream_t stream);

// W4A16 fused projection for M >= 17 on tcgen05 (weights as the TMEM operand).
cudaError_t launch_tc_w4a16(const __half* x, const uint32_t* const w[3], const __half* const s[3],
                            __half* const out[3], int M, int N, int K, int num_sms,
                            cudaStream_t stream);
// W8A16 prefill: packed INT8 weights u32[K/4, N] (byte i = K-row 4r+i), one
// f32 scale per projection.
cudaError_t launch_tc_w8a16(const __half* x, const uint32_t* const w[3], const float scale[3],
                            __half* const out[3], int M, int N, int K, int num_sms,
                            cudaStream_t stream);

// Bit-exact dequantisation (debug / test entry).
cudaError_t launch_dequant_debug(const uint32_t* w, const __half* s, __half* out, int K, int N,
                                 int variant, cudaStream_t stream);

// Device error word (bounded-wait timeouts), read and cleared by the host API.
constexpr unsigned kDevErrTimeoutHost = 1u;   // same bit as kDevErrTimeout in kaio_device.cuh
unsigned read_and_clear_tc_errors();

// Raise a kernel's dynamic shared memory limit once per (kernel, device):
// later calls (including those made while a stream is being captured into a
// CUDA graph) only look the pair up.
cudaError_t ensure_smem_limit(const void* kernel, int bytes);

// Driver entry point for tensor-map encoding (resolved once through the runtime).
CUresult encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                              uint64_t inner, uint64_t outer, uint64_t row_bytes,
                              uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz);

}  // namespace kaio
