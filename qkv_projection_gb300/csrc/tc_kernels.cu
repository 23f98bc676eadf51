// tcgen05 (5th-generation tensor core) kernels of libkaio_qkv:
//
//  * tc_gemm_kernel: dense f16 x f16 -> f32, C = Aop * Bop, for
//    "kaio-candle 0.2.0 -- src/matmul_tc_async.rs" (forward, and the backward
//    dA = grad * B^T, dB = A^T * grad of MatmulTcAsyncOp::bwd, taken here by
//    reading the stored operands in the other major order instead of copying
//    transposes).
//  * tc_qkv_prefill_kernel<4>: the W4A16 fused QKV projection of
//    "kaio-candle -- src/qkv_project_int4.rs" for M >= 17;
//    tc_qkv_prefill_kernel<8>: its INT8 sibling (W8A16), named in the module
//    doc of that page; INT4 packing with 8-bit fields and one f32 scale per
//    projection, applied to the f32 accumulator in the epilogue.
//
// Both share one pipeline shape: a TMA producer warp fills a ring of shared
// memory stages, MMA-issuing threads (one; in the projection kernel one per
// projection) issue tcgen05.mma into f32 accumulators in tensor memory, and
// the remaining warps drain the accumulators with
// tcgen05.ld and write the outputs. Every wait on an mbarrier is bounded.
//
// Dense: A and B both come from shared memory (128B-swizzled TMA tiles);
// 128 x 256 output tile; two accumulator buffers so the epilogue of one tile
// overlaps the main loop of the next.
//
// W4A16 / W8A16: the product is computed transposed, D_p[n, m] = Wd_p^T[n, :] x^T[:, m],
// so that the dequantised weights are the MMA's A operand and can live in
// tensor memory: eight dequant warps read packed words from the staged tile,
// build f16 operands in registers and write them to TMEM with tcgen05.st; the
// shared activation tile x is the B operand and is read once per k-step for all
// three projections. No dequantised weight ever touches shared memory.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <map>
#include <mutex>
#include <unordered_map>
#include <utility>

#include "kaio_device.cuh"
#include "kaio_internal.h"

namespace kaio {

__device__ unsigned g_tc_err = 0;

namespace {

// ============================================================== dense GEMM
// A CTA pair computes a 256-row tile of C with tcgen05.mma of M = 256 per 16 K
// (cta_group::2): CTA rank r loads A rows m0 + 128r .. +127 into its own
// shared memory and holds C rows m0 + 128r .. +127 in its tensor memory. Each
// MMA has N = 256 columns, of which each CTA supplies 128 from its shared
// memory, so every B column is read once per pair.
//
// Two tile widths (the host picks per call):
//  * wide: 512 columns, two MMAs per 16 K into the CTA's whole 512-column
//    TMEM. Each CTA takes 48 KB per 64-K step for 2 x 128 x 512 x 64 FLOPs,
//    a quarter fewer bytes per FLOP than 256 columns; used when the wide tiles
//    fill at least one wave of CTA pairs.
//  * narrow: 256 columns, one MMA per 16 K into one of two 256-column TMEM
//    buffers, so a tile's epilogue overlaps the next tile's main loop.
// The epilogue stages each 128-byte-wide column chunk of the CTA's rows in
// shared memory (128B-swizzled) and writes it with a TMA store; a wide tile's
// TMEM is handed back as soon as its last chunk has been read, while the
// stores drain on their own. (Row-per-thread global stores of the same data
// cost a wide tile ~20 % of its time.)
constexpr int GBM = 128;                       // rows of A (and of C) per CTA
constexpr int GBK = 64;
constexpr int GA_BYTES = GBM * GBK * 2;        // 16 KB
constexpr int GB_PIECE = 128 * GBK * 2;        // 16 KB: 128 columns of B for one MMA
constexpr int GMAX_STAGES = 6;
constexpr int GTHREADS = 224;                  // w0, w6 TMA; w1 MMA (rank 0) + TMEM; w2..5 epilogue
constexpr uint32_t GTMEM_COLS = 512;
constexpr int GOUT_BUF = 128 * 128;            // one staged output chunk: 128 rows x 128 bytes
constexpr size_t GSMEM = static_cast<size_t>(GMAX_STAGES) * (GA_BYTES + GB_PIECE) + 2 * GOUT_BUF + 1024;

template <bool kWide>
struct GShape {
  static constexpr int kN = kWide ? 512 : 256;           // columns of C per pair tile
  static constexpr int kPieces = kN / 256;                // MMAs per 16 K
  static constexpr int kStageBytes = GA_BYTES + kPieces * GB_PIECE;
  static constexpr int kStages = kWide ? 4 : 6;
  static constexpr int kBufs = kWide ? 1 : 2;             // TMEM accumulators of kN columns
  static_assert(kStages % 2 == 0, "the two producers own alternate stages");
  static_assert(kStages * kStageBytes + 2 * GOUT_BUF + 1024 <= GSMEM, "shared memory");
};

struct GemmParams {
  void* c;              // f32 or f16 [M, N]
  int M, N, K;
  int m_pairs, tiles;   // 256-row blocks; pair tiles
};

// TMA store of one box from shared memory (bulk-group completion), and the
// waits on this thread's outstanding bulk groups.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(map),
               "r"(smem_u32(src)), "r"(c0), "r"(c1)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// at most one group still reading its shared-memory source
__device__ __forceinline__ void bulk_wait_read1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// every group complete (its writes performed)
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Named barrier that also ANDs a flag over its `count` threads, so that they
// all take the same branch afterwards.
__device__ __forceinline__ bool named_and(int id, int count, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.and.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// C16: the epilogue rounds the f32 accumulators to f16 (round-to-nearest-even)
// and stores f16, fusing the cast the page's backward applies afterwards.
//
// Barriers: both CTAs' stage bytes are counted on rank 0's full[st] (rank 0's
// producer expects them all; the pair form of the TMA load lets rank 1's
// copies complete there); rank 0's MMA thread releases stage st in both CTAs and hands each CTA its accumulator with
// commits to each CTA's own barriers; both CTAs' epilogue warps arrive on rank
// 0's acc_empty. Persistent: pair p takes tiles p, p + pairs, ...; tiles are
// numbered down the rows first, so the pairs running at one time share B tiles
// through L2.
template <bool A_MN, bool B_MN, bool C16, bool kWide>
__global__ void __launch_bounds__(GTHREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
  using S = GShape<kWide>;
  constexpr int kStages = S::kStages, kStageBytes = S::kStageBytes;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = align_smem_1024(smem_raw);
  unsigned char* out_stage = smem + kStages * kStageBytes;    // two 16 KB output chunks, 1024-aligned
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages], acc_full[2], acc_empty[2], mma_done;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_ctarank());
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);                  // rank 0's: its producer's expect_tx for both CTAs' bytes
      mbar_init(&empty[s], 1);                 // rank 0's MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);              // rank 0's MMA commit
      mbar_init(&acc_empty[b], 8);             // rank 0's: 4 epilogue warps of each CTA
    }
    mbar_init(&mma_done, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(&tmem_base_sh, GTMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncwarp();
  cluster_sync_all();                          // both CTAs' barriers exist before any remote use
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const int nk = (p.K + GBK - 1) / GBK;
  volatile int* abort = &abort_flag;
  const int pair = static_cast<int>(blockIdx.x) >> 1;
  const int pstride = static_cast<int>(gridDim.x) >> 1;
  // rank 0's copy of a barrier of this CTA, and the peer's copy
  auto at_rank0 = [&](uint64_t* bar) { return dsmem_map(smem_u32(bar), 0); };
  auto at_peer = [&](uint64_t* bar) { return dsmem_map(smem_u32(bar), static_cast<uint32_t>(rank ^ 1)); };

  if (warp == 0 || warp == 6) {
    // Two producer threads, one per warp, take alternate k-steps (and so
    // alternate stages): a thread spends several hundred cycles per stage on
    // its barrier operations and copies, and two of them keep the ring full.
    if (lane == 0) {
      const int pid = warp == 0 ? 0 : 1;
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      int st = 0;
      uint32_t ph = 0;
      uint32_t fills[kStages] = {};
      for (int t = pair; t < p.tiles; t += pstride) {
        const int m0 = (t % p.m_pairs) * (2 * GBM) + rank * GBM;
        // this CTA's 128 columns of MMA j start at n0 + 256 j
        const int n0 = (t / p.m_pairs) * S::kN + rank * 128;
        for (int kb = 0; kb < nk; ++kb) {
          if ((st & 1) != pid) {                 // the other producer's stage
            if (++st == kStages) { st = 0; ph ^= 1; }
            continue;
          }
          if (!mbar_wait_cluster(&empty[st], ph ^ 1, abort, &g_tc_err)) goto producer_done;
          ++fills[st];
          unsigned char* sa = smem + st * kStageBytes;
          unsigned char* sb = sa + GA_BYTES;
          // Only rank 0's producer arrives (expecting both CTAs' bytes); rank
          // 1's copies count their bytes on rank 0's barrier directly. A
          // thread's arrive on another CTA's barrier stalls it for about as long
          // as a k-step takes, so no thread makes one per k-step.
          const uint32_t fb = at_rank0(&full[st]);
          if (rank == 0) mbar_arrive_expect_tx(&full[st], 2 * kStageBytes);
          if (!A_MN) {
            tma_load_2d_pair(sa, &tmA, fb, kb * GBK, m0);
          } else {
            tma_load_2d_pair(sa, &tmA, fb, m0, kb * GBK);
            tma_load_2d_pair(sa + 8192, &tmA, fb, m0 + 64, kb * GBK);
          }
#pragma unroll
          for (int j = 0; j < S::kPieces; ++j) {
            if (!B_MN) {
              tma_load_2d_pair(sb + j * GB_PIECE, &tmB, fb, kb * GBK, n0 + 256 * j);
            } else {
              tma_load_2d_pair(sb + j * GB_PIECE, &tmB, fb, n0 + 256 * j, kb * GBK);
              tma_load_2d_pair(sb + j * GB_PIECE + 8192, &tmB, fb, n0 + 256 * j + 64, kb * GBK);
            }
          }
          if (++st == kStages) { st = 0; ph ^= 1; }
        }
      }
    producer_done:
      // No copy may still be landing in this CTA's shared memory when it
      // exits: every fill is consumed by an MMA (which waited for its bytes)
      // before its release reaches this CTA's stage.
      for (int s2 = 0; s2 < kStages; ++s2)
        if (fills[s2]) mbar_wait_cluster_drain(&empty[s2], (fills[s2] - 1) & 1, &g_tc_err);
    }
  } else if (warp == 1) {
    if (rank == 0 && lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(2 * GBM, 256, A_MN, B_MN);
      int st = 0;
      uint32_t ph = 0;
      int buf = 0;
      uint32_t aph = 0;
      for (int t = pair; t < p.tiles; t += pstride) {
        if (!mbar_wait_cluster(&acc_empty[buf], aph ^ 1, abort, &g_tc_err)) break;
        tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(buf * S::kN);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_cluster(&full[st], ph, abort, &g_tc_err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + st * kStageBytes);
          const uint32_t sb = sa + GA_BYTES;
#pragma unroll
          for (int kk = 0; kk < GBK / 16; ++kk) {
            const uint64_t ad = A_MN ? sdesc_sw128(sa + kk * 2048, 8192, 1024)
                                     : sdesc_sw128(sa + kk * 32, 16, 1024);
#pragma unroll
            for (int j = 0; j < S::kPieces; ++j) {
              const uint32_t bj = sb + j * GB_PIECE;
              const uint64_t bd = B_MN ? sdesc_sw128(bj + kk * 2048, 8192, 1024)
                                       : sdesc_sw128(bj + kk * 32, 16, 1024);
              umma_ss_pair(d + 256 * j, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
            }
          }
          umma_commit_pair(smem_u32(&empty[st]));
          umma_commit_pair(at_peer(&empty[st]));
          if (++st == kStages) { st = 0; ph ^= 1; }
        }
        if (!ok) break;
        umma_commit_pair(smem_u32(&acc_full[buf]));
        umma_commit_pair(at_peer(&acc_full[buf]));
        if (++buf == S::kBufs) { buf = 0; aph ^= 1; }
      }
      // Every MMA issued (and with it every commit to either CTA) has
      // completed before TMEM is released.
      umma_commit_pair(smem_u32(&mma_done));
      mbar_wait_cluster_drain(&mma_done, 0, &g_tc_err);
    }
  } else if (warp <= 5) {
    // Epilogue: warp w drains TMEM lanes 32*(w%4) .. +31 (this CTA's rows) in
    // chunks of 128 bytes per row (32 f32 or 64 f16 columns): TMEM ->
    // registers -> a 128B-swizzled 16 KB staging buffer (two, alternating) ->
    // one TMA store per chunk, issued by warp 2's lane 0 once all four warps
    // have written it. TMA clips rows >= M and columns >= N.
    constexpr int kChunkCols = C16 ? 64 : 32;
    constexpr int kChunks = S::kN / kChunkCols;
    const bool issuer = warp == 2 && lane == 0;
    const int sp = warp & 3;
    const int row = 32 * sp + lane;             // row of the CTA's 128 in the chunk
    const uint32_t row_tmem = static_cast<uint32_t>(32 * sp) << 16;
    int buf = 0, ob = 0, nstored = 0;
    uint32_t aph = 0;
    for (int t = pair; t < p.tiles; t += pstride) {
      const int m0 = (t % p.m_pairs) * (2 * GBM) + rank * GBM, n0 = (t / p.m_pairs) * S::kN;
      // the four warps meet at named barriers below: they leave together
      const bool got = mbar_wait_cluster(&acc_full[buf], aph, abort, &g_tc_err);
      if (!named_and(1, 128, got)) break;
      tc_fence_after();
#pragma unroll 1
      for (int ch = 0; ch < kChunks; ++ch) {
        uint32_t r[kChunkCols];
        if constexpr (C16) {
          uint32_t lo[32], hi[32];
          tmem_ld32(tmem + row_tmem + buf * S::kN + ch * 64, lo);
          tmem_ld32(tmem + row_tmem + buf * S::kN + ch * 64 + 32, hi);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const __half2 a2 = __floats2half2_rn(__uint_as_float(lo[2 * i]), __uint_as_float(lo[2 * i + 1]));
            const __half2 b2 = __floats2half2_rn(__uint_as_float(hi[2 * i]), __uint_as_float(hi[2 * i + 1]));
            r[i] = *reinterpret_cast<const uint32_t*>(&a2);
            r[16 + i] = *reinterpret_cast<const uint32_t*>(&b2);
          }
        } else {
          tmem_ld32(tmem + row_tmem + buf * S::kN + ch * 32, r);
          tmem_ld_wait();
        }
        if (ch == kChunks - 1) {
          // the whole accumulator has been read: hand it back to the MMAs
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(at_rank0(&acc_empty[buf]));
        }
        // staging buffer ob is free once the store issued from it two chunks
        // ago has read it
        if (issuer && nstored >= 2) bulk_wait_read1();
        named_sync(1, 128);
        unsigned char* dst = out_stage + ob * GOUT_BUF + row * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 v = make_uint4(r[4 * u], r[4 * u + 1], r[4 * u + 2], r[4 * u + 3]);
          *reinterpret_cast<uint4*>(dst + ((u ^ (row & 7)) << 4)) = v;
        }
        fence_proxy_async_smem();
        named_sync(1, 128);
        if (issuer) {
          // a box wholly outside C writes nothing; its group is committed
          // (empty) all the same, so that the group two back is always the
          // store that last read this staging buffer
          if (m0 < p.M && n0 + ch * kChunkCols < p.N)
            tma_store_2d(&tmC, out_stage + ob * GOUT_BUF, n0 + ch * kChunkCols, m0);
          bulk_commit();
        }
        ++nstored;
        ob ^= 1;
      }
      if (++buf == S::kBufs) { buf = 0; aph ^= 1; }
    }
    if (issuer) bulk_wait_all();                // every store done before the CTA exits
  }

  tc_fence_before();
  __syncwarp();
  cluster_sync_all();                          // no remote arrive or commit targets an exited CTA
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem, GTMEM_COLS);
  }
}

// ============================================================ W4A16 prefill
constexpr int PBM = 128;                 // x rows per tile        (MMA N)
constexpr int PBN = 128;                 // output columns per tile (MMA M)
constexpr int PBK = 64;                  // K per TMA stage
constexpr int PSTAGES = 4;
constexpr int PX_BYTES = PBM * PBK * 2;          // 16384
constexpr int PMMA_WARPS = 3;                    // one MMA-issuing warp per projection
constexpr int PDQ_WARPS = 8;
constexpr int PTHREADS = (1 + PMMA_WARPS + PDQ_WARPS) * 32;   // w0 TMA, w1..3 MMA, w4..11 dequant + epilogue
constexpr uint32_t PTMEM_COLS = 512;
constexpr uint32_t PA_COL0 = 384;                // A stages after the three accumulators
constexpr uint32_t PA_STAGE_COLS = 48;           // 3 projections x 16 columns (32 K)

// Stage layout of one weight format (kBits = 4: INT4 with f16 group scales;
// kBits = 8: INT8 with one f32 scale per projection, applied in the epilogue).
template <int kBits>
struct PFmt {
  static constexpr int kRows = PBK * kBits / 32;             // packed rows per stage: 8 or 16
  static constexpr int kWBytes = kRows * PBN * 4;            // one projection's words: 4 or 8 KB
  static constexpr int kSBytes = kBits == 4 ? PBN * 2 : 0;   // one projection's scale row
  static constexpr int kTx = PX_BYTES + 3 * kWBytes + 3 * kSBytes;   // bytes landed per stage
  static constexpr int kStage = kBits == 4 ? 30720 : 40960;  // padded: x tiles stay 1024-aligned
  static constexpr size_t kSmem = static_cast<size_t>(PSTAGES) * kStage + 1024;
  static_assert(kTx <= kStage && kStage % 1024 == 0, "stage layout");
};

struct PrefillParams {
  __half* out[3];
  float scale[3];        // INT8: per-projection scales
  int M, N, K;
  int m_blocks, tiles;
};

template <int kBits>
__global__ void __launch_bounds__(PTHREADS, 1)
    tc_qkv_prefill_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW0,
                    const __grid_constant__ CUtensorMap tmW1, const __grid_constant__ CUtensorMap tmW2,
                    const __grid_constant__ CUtensorMap tmS0, const __grid_constant__ CUtensorMap tmS1,
                    const __grid_constant__ CUtensorMap tmS2, const PrefillParams p) {
  using F = PFmt<kBits>;
  constexpr int PW_BYTES = F::kWBytes, PS_BYTES = F::kSBytes, PSTAGE_BYTES = F::kStage;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = align_smem_1024(smem_raw);
  __shared__ __align__(8) uint64_t full[PSTAGES], empty[PSTAGES], a_full[2], a_empty[2],
      acc_full, acc_empty, mma_done[PMMA_WARPS];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < PSTAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1 + PDQ_WARPS);  // every dequant warp + the release after the MMAs
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&a_full[a], PDQ_WARPS);
      mbar_init(&a_empty[a], PMMA_WARPS);   // one commit per MMA warp
    }
    mbar_init(&acc_full, PMMA_WARPS);
    mbar_init(&acc_empty, PDQ_WARPS);
    for (int w = 0; w < PMMA_WARPS; ++w) mbar_init(&mma_done[w], 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, PTMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const int nks = p.K / PBK;   // K is a multiple of 128
  volatile int* abort = &abort_flag;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tmX);
      tma_prefetch_desc(&tmW0); tma_prefetch_desc(&tmW1); tma_prefetch_desc(&tmW2);
      if constexpr (kBits == 4) {
        tma_prefetch_desc(&tmS0); tma_prefetch_desc(&tmS1); tma_prefetch_desc(&tmS2);
      }
      int st = 0;
      uint32_t ph = 0;
      uint32_t fills[PSTAGES] = {0, 0, 0, 0};
      for (int tile = blockIdx.x; tile < p.tiles; tile += gridDim.x) {
        const int m0 = (tile % p.m_blocks) * PBM, n0 = (tile / p.m_blocks) * PBN;
        for (int ks = 0; ks < nks; ++ks) {
          if (!mbar_wait(&empty[st], ph ^ 1, abort, &g_tc_err)) goto producer_done;
          ++fills[st];
          unsigned char* sx = smem + st * PSTAGE_BYTES;
          mbar_arrive_expect_tx(&full[st], F::kTx);
          tma_load_2d(sx, &tmX, &full[st], ks * PBK, m0);
          unsigned char* sw = sx + PX_BYTES;
          tma_load_2d(sw, &tmW0, &full[st], n0, ks * F::kRows);
          tma_load_2d(sw + PW_BYTES, &tmW1, &full[st], n0, ks * F::kRows);
          tma_load_2d(sw + 2 * PW_BYTES, &tmW2, &full[st], n0, ks * F::kRows);
          if constexpr (kBits == 4) {
            unsigned char* ss = sx + PX_BYTES + 3 * PW_BYTES;
            tma_load_2d(ss, &tmS0, &full[st], n0, ks >> 1);
            tma_load_2d(ss + PS_BYTES, &tmS1, &full[st], n0, ks >> 1);
            tma_load_2d(ss + 2 * PS_BYTES, &tmS2, &full[st], n0, ks >> 1);
          }
          if (++st == PSTAGES) { st = 0; ph ^= 1; }
        }
      }
    producer_done:
      for (int s2 = 0; s2 < PSTAGES; ++s2)
        if (fills[s2]) mbar_wait_drain(&full[s2], (fills[s2] - 1) & 1, &g_tc_err);
    }
  } else if (warp <= PMMA_WARPS) {
    // MMA warp q issues projection q's MMAs into its accumulator D[q]; three
    // issuing warps overlap one another's barrier waits and commits with MMAs.
    // No wait on the shared-memory stage itself: an A stage is full only after
    // the dequant warps have waited for the stage, so it has landed. These
    // warps do nothing but wait for A stages, issue and commit them: they
    // release no shared-memory stage (the dequant warps do, below) and test no
    // barrier ahead -- each such operation costs the issuing thread 150-300
    // cycles between MMAs.
    const int q = warp - 1;
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(PBN, PBM, false, false);
      int st = 0, a = 0;
      uint32_t aph = 0, cph = 0;
      for (int tile = blockIdx.x; tile < p.tiles; tile += gridDim.x) {
        if (!mbar_wait(&acc_empty, cph ^ 1, abort, &g_tc_err)) break;
        tc_fence_after();
        bool ok = true;
        for (int ks = 0; ks < nks && ok; ++ks) {
          const uint64_t bd0 = sdesc_sw128(smem_u32(smem + st * PSTAGE_BYTES), 16, 1024);
          const uint32_t blo = static_cast<uint32_t>(bd0), bhi = static_cast<uint32_t>(bd0 >> 32);
          for (int hh = 0; hh < 2; ++hh) {
            if (!mbar_wait(&a_full[a], aph, abort, &g_tc_err)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
              const uint32_t at = tmem + PA_COL0 + a * PA_STAGE_COLS + q * 16 + kk * 8;
              umma_ts_lohi(tmem + q * PBM, at, blo + (((2 * hh + kk) * 32) >> 4), bhi, idesc,
                           (ks | hh | kk) != 0 ? 1u : 0u);
            }
            umma_commit(&a_empty[a]);
            if (++a == 2) { a = 0; aph ^= 1; }
          }
          if (!ok) break;
          if (++st == PSTAGES) st = 0;
        }
        if (!ok) break;
        umma_commit(&acc_full);
        cph ^= 1;
      }
      umma_commit(&mma_done[q]);
      mbar_wait_drain(&mma_done[q], 0, &g_tc_err);
    }
  } else {
    // Dequant + epilogue warps. TMEM lane group sp = warp % 4: this thread owns
    // output column n0 + 32*sp + lane (TMEM lane = A row = column). hf picks the
    // 16 K of each 32-K A stage this warp fills (two INT4 or four INT8 packed
    // rows), and the half of the x rows it drains in the epilogue.
    const int sp = warp & 3;
    const int hf = (warp - 1 - PMMA_WARPS) >> 2;
    const int nl = 32 * sp + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * sp) << 16;
    int st = 0, a = 0;
    int rel_st = -1;   // shared-memory stage of the previous k-step, not yet released
    uint32_t ph = 0, aph = 0, cph = 0;
    for (int tile = blockIdx.x; tile < p.tiles; tile += gridDim.x) {
      const int m0 = (tile % p.m_blocks) * PBM, n0 = (tile / p.m_blocks) * PBN;
      bool ok = true;
      for (int ks = 0; ks < nks && ok; ++ks) {
        if (!mbar_wait(&full[st], ph, abort, &g_tc_err)) { ok = false; break; }
        const unsigned char* sx = smem + st * PSTAGE_BYTES;
        const uint32_t* sw = reinterpret_cast<const uint32_t*>(sx + PX_BYTES);
        const __half* ss = reinterpret_cast<const __half*>(sx + PX_BYTES + 3 * PW_BYTES);
        uint32_t s2[3];
#pragma unroll
        for (int q = 0; q < 3; ++q) {
          if constexpr (kBits == 4) {
            const uint16_t sb = __half_as_ushort(ss[q * PBN + nl]);
            s2[q] = half2_bits(sb, sb);
          } else {
            s2[q] = 0;
          }
        }
        (void)ss;
        // Each half's 16 K of this warp are converted into registers before
        // the wait for their A stage: only the stores need the stage, so the
        // conversion overlaps the MMAs still reading it. INT4 converts both
        // halves up front, so that nothing but a wait and the stores sits
        // between the two halves' hand-offs (W4A16 4096^3: 317.5 -> 312 us);
        // the INT8 conversion is short enough that this measured slower
        // (285 -> 295 us), so it converts one half at a time. Column
        // q*16 + hf*8 + c of an A stage holds K pair c of this warp's 16 K of
        // projection q.
        uint32_t v[2][3][8];
        auto convert_half = [&](const int hh) {
#pragma unroll
          for (int q = 0; q < 3; ++q) {
            if constexpr (kBits == 4) {
              const int r0 = hh * 4 + hf * 2;
              const uint32_t w0 = sw[q * (PW_BYTES / 4) + r0 * PBN + nl];
              const uint32_t w1 = sw[q * (PW_BYTES / 4) + (r0 + 1) * PBN + nl];
              uint32_t v0[4], v1[4];
              dequant_natural(w0, s2[q], v0);
              dequant_natural(w1, s2[q], v1);
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                v[hh][q][c] = v0[c];
                v[hh][q][4 + c] = v1[c];
              }
            } else {
              const int r0 = hh * 8 + hf * 4;
#pragma unroll
              for (int j = 0; j < 4; ++j)
                int8x4_to_half2x2(sw[q * (PW_BYTES / 4) + (r0 + j) * PBN + nl], v[hh][q][2 * j],
                                  v[hh][q][2 * j + 1]);
            }
          }
        };
        if constexpr (kBits == 4) {
          convert_half(0);
          convert_half(1);
          // Pin the conversion here: left alone, the compiler sinks each
          // half's arithmetic to its stores, after the barrier wait.
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int q = 0; q < 3; ++q)
#pragma unroll
              for (int c = 0; c < 8; ++c) asm volatile("" : "+r"(v[hh][q][c]));
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          if constexpr (kBits == 8) convert_half(hh);
          if (!mbar_wait(&a_empty[a], aph ^ 1, abort, &g_tc_err)) { ok = false; break; }
          // A stage 1 is free once the MMAs of the previous k-step's second
          // half have completed, i.e. every MMA reading that k-step's x tile:
          // one warp releases its shared-memory stage on the MMA's behalf.
          if (hh == 1 && rel_st >= 0 && warp == 1 + PMMA_WARPS && lane == 0) mbar_arrive(&empty[rel_st]);
          tc_fence_after();
#pragma unroll
          for (int q = 0; q < 3; ++q)
            tmem_st8(tmem + lane_base + PA_COL0 + a * PA_STAGE_COLS + q * 16 + hf * 8, v[hh][q]);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&a_full[a]);
          if (++a == 2) { a = 0; aph ^= 1; }
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
        rel_st = st;
        if (++st == PSTAGES) { st = 0; ph ^= 1; }
      }
      if (!ok) break;

      // Epilogue: D_q[n][m] -> out_q[m0 + m][n0 + n] as f16.
      if (!mbar_wait(&acc_full, cph, abort, &g_tc_err)) break;
      tc_fence_after();
      const int n = n0 + nl;
      const bool odd = lane & 1;
      const int ncol = n0 + (nl & ~1);
#pragma unroll 1
      for (int q = 0; q < 3; ++q) {
        __half* out = (q == 0) ? p.out[0] : (q == 1) ? p.out[1] : p.out[2];
        const float sc = (q == 0) ? p.scale[0] : (q == 1) ? p.scale[1] : p.scale[2];
#pragma unroll 1
        for (int mh = 0; mh < 2; ++mh) {
          const int mb = 64 * hf + 32 * mh;
          uint32_t r[32];
          tmem_ld32(tmem + lane_base + q * PBM + mb, r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            float own_lo = __uint_as_float(r[j]), own_hi = __uint_as_float(r[j + 1]);
            if constexpr (kBits == 8) {
              own_lo *= sc;
              own_hi *= sc;
            }
            const float send = odd ? own_lo : own_hi;
            const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
            const int m = m0 + mb + j + (odd ? 1 : 0);
            const __half2 h = odd ? __floats2half2_rn(recv, own_hi) : __floats2half2_rn(own_lo, recv);
            if (m < p.M && ncol < p.N)
              *reinterpret_cast<__half2*>(out + static_cast<size_t>(m) * p.N + ncol) = h;
          }
        }
      }
      (void)n;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty);
      cph ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, PTMEM_COLS);
  }
}

// ============================================================ debug dequant
__global__ void dequant_debug_kernel(const uint32_t* __restrict__ w, const __half* __restrict__ s,
                                     __half* __restrict__ out, int K, int N, int variant) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long total = static_cast<long long>(K / 8) * N;
  if (idx >= total) return;
  const int r = static_cast<int>(idx / N), n = static_cast<int>(idx % N);
  const uint32_t word = w[idx];
  const uint16_t sb = __half_as_ushort(s[static_cast<size_t>(r / 16) * N + n]);
  const uint32_t s2 = half2_bits(sb, sb);
  uint16_t vals[8];
  if (variant == 0) {
    uint32_t o[4];
    dequant_natural(word, s2, o);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      vals[2 * c] = static_cast<uint16_t>(o[c] & 0xFFFFu);
      vals[2 * c + 1] = static_cast<uint16_t>(o[c] >> 16);
    }
  } else {
    const PairedNibbles pn(word);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t v = pn.pair(j, s2);
      vals[j] = static_cast<uint16_t>(v & 0xFFFFu);
      vals[j + 4] = static_cast<uint16_t>(v >> 16);
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i)
    out[static_cast<size_t>(8 * r + i) * N + n] = __ushort_as_half(vals[i]);
}

}  // namespace

// ================================================================== host side
namespace {
// One encoded tensor map per distinct set of arguments, per host thread: a
// map depends only on these values, and weights (and often activation
// buffers) are the same from call to call. Encoding costs the calling thread
// about as much as the rest of a decode call's host work together.
struct TmKey {
  uint64_t base, inner, outer, row_bytes;
  uint32_t box_inner, box_outer, dtype, swz;
  bool operator==(const TmKey& o) const {
    return base == o.base && inner == o.inner && outer == o.outer && row_bytes == o.row_bytes &&
           box_inner == o.box_inner && box_outer == o.box_outer && dtype == o.dtype && swz == o.swz;
  }
};
struct TmKeyHash {
  size_t operator()(const TmKey& k) const {
    uint64_t h = k.base * 0x9E3779B97F4A7C15ull;
    for (uint64_t v : {k.inner, k.outer, k.row_bytes,
                       (static_cast<uint64_t>(k.box_inner) << 32) | k.box_outer,
                       (static_cast<uint64_t>(k.dtype) << 32) | k.swz})
      h = (h ^ v) * 0x100000001B3ull;
    return static_cast<size_t>(h ^ (h >> 29));
  }
};
constexpr size_t kTmCacheMax = 512;   // entries per host thread before the cache is emptied
}  // namespace

CUresult encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                              uint64_t inner, uint64_t outer, uint64_t row_bytes,
                              uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  if (!fn) return CUDA_ERROR_NOT_FOUND;
  thread_local std::unordered_map<TmKey, CUtensorMap, TmKeyHash> cache;
  const TmKey key{reinterpret_cast<uint64_t>(base), inner, outer, row_bytes, box_inner, box_outer,
                  static_cast<uint32_t>(dtype), static_cast<uint32_t>(swz)};
  auto it = cache.find(key);
  if (it != cache.end()) {
    *map = it->second;
    return CUDA_SUCCESS;
  }
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r == CUDA_SUCCESS) {
    if (cache.size() >= kTmCacheMax) cache.clear();
    cache.emplace(key, *map);
  }
  return r;
}

cudaError_t ensure_smem_limit(const void* kernel, int bytes) {
  // The attribute is one upper bound per (kernel, device): only ever raise it,
  // so that a launch needing less never lowers it under an earlier, larger need.
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  // A per-thread record of limits already in place spares the lock on every call.
  thread_local std::map<std::pair<const void*, int>, int> seen;
  auto hit = seen.find(std::make_pair(kernel, dev));
  if (hit != seen.end() && bytes <= hit->second) return cudaSuccess;
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> limit;
  std::lock_guard<std::mutex> lk(mu);
  int& cur = limit[std::make_pair(kernel, dev)];
  if (bytes <= cur) {
    seen[std::make_pair(kernel, dev)] = cur;
    return cudaSuccess;
  }
  cudaFuncAttributes fa{};
  e = cudaFuncGetAttributes(&fa, kernel);
  if (e != cudaSuccess) return e;
  if (fa.maxDynamicSharedSizeBytes >= bytes) {
    cur = fa.maxDynamicSharedSizeBytes;
    seen[std::make_pair(kernel, dev)] = cur;
    return cudaSuccess;
  }
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) {
    cur = bytes;
    seen[std::make_pair(kernel, dev)] = cur;
  }
  return e;
}

static cudaError_t map_error(CUresult r) {
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

namespace {
// Resident clusters of two GEMM CTAs on device `dev` (cached per kernel).
int gemm_max_active_pairs(const void* kern, int dev) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> cache;
  std::lock_guard<std::mutex> lk(mu);
  const auto key = std::make_pair(kern, dev);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(GTHREADS);
  cfg.dynamicSmemBytes = GSMEM;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  cache[key] = n;
  return n;
}
}  // namespace

cudaError_t launch_tc_gemm(const void* a, const void* b, void* c, GemmShape sh, bool a_mn,
                           bool b_mn, bool c_f16, int num_sms, cudaStream_t stream) {
  CUtensorMap ta, tb;
  CUresult r;
  // Aop is [M x K]; stored [M][K] (K-major) or [K][M] (MN-major).
  if (!a_mn)
    r = encode_tensor_map_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a, sh.K, sh.M,
                             static_cast<uint64_t>(sh.K) * 2, GBK, GBM, CU_TENSOR_MAP_SWIZZLE_128B);
  else
    r = encode_tensor_map_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a, sh.M, sh.K,
                             static_cast<uint64_t>(sh.M) * 2, 64, GBK, CU_TENSOR_MAP_SWIZZLE_128B);
  if (r != CUDA_SUCCESS) return map_error(r);
  // Bop is [K x N]; stored [N][K] (K-major) or [K][N] (MN-major). Each CTA of
  // a pair loads 128 columns per MMA: one 128-row K-major box, or two
  // 64-column MN-major boxes.
  if (!b_mn)
    r = encode_tensor_map_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, b, sh.K, sh.N,
                             static_cast<uint64_t>(sh.K) * 2, GBK, 128, CU_TENSOR_MAP_SWIZZLE_128B);
  else
    r = encode_tensor_map_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, b, sh.N, sh.K,
                             static_cast<uint64_t>(sh.N) * 2, 64, GBK, CU_TENSOR_MAP_SWIZZLE_128B);
  if (r != CUDA_SUCCESS) return map_error(r);
  // C [M][N] f32 or f16, stored by the epilogue in 128-row x 128-byte boxes.
  CUtensorMap tc;
  if (c_f16)
    r = encode_tensor_map_2d(&tc, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, c, sh.N, sh.M,
                             static_cast<uint64_t>(sh.N) * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
  else
    r = encode_tensor_map_2d(&tc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, c, sh.N, sh.M,
                             static_cast<uint64_t>(sh.N) * 4, 32, 128, CU_TENSOR_MAP_SWIZZLE_128B);
  if (r != CUDA_SUCCESS) return map_error(r);

  GemmParams p{};
  p.c = c;
  p.M = sh.M;
  p.N = sh.N;
  p.K = sh.K;
  p.m_pairs = (sh.M + 2 * GBM - 1) / (2 * GBM);

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  auto pick = [&](bool wide) -> const void* {
#define KAIO_PICK_GEMM(AM, BM_, W)                                                                      \
  return c_f16 ? reinterpret_cast<const void*>(tc_gemm_kernel<AM, BM_, true, W>)                        \
               : reinterpret_cast<const void*>(tc_gemm_kernel<AM, BM_, false, W>)
    if (wide) {
      if (!a_mn && b_mn) KAIO_PICK_GEMM(false, true, true);
      if (!a_mn && !b_mn) KAIO_PICK_GEMM(false, false, true);
      if (a_mn && b_mn) KAIO_PICK_GEMM(true, true, true);
      KAIO_PICK_GEMM(true, false, true);
    }
    if (!a_mn && b_mn) KAIO_PICK_GEMM(false, true, false);
    if (!a_mn && !b_mn) KAIO_PICK_GEMM(false, false, false);
    if (a_mn && b_mn) KAIO_PICK_GEMM(true, true, false);
    KAIO_PICK_GEMM(true, false, false);
#undef KAIO_PICK_GEMM
  };
  // Wide (512-column) tiles when they fill at least one wave of resident CTA
  // pairs (a pair sits in one GPC); narrow ones otherwise, so that small
  // problems spread over more SMs.
  const void* kern = pick(true);
  int slots = gemm_max_active_pairs(kern, dev);
  if (slots <= 0) slots = num_sms / 2;
  const int wide_tiles = p.m_pairs * ((sh.N + 511) / 512);
  const bool wide = wide_tiles >= slots;
  if (!wide) {
    kern = pick(false);
    const int s2 = gemm_max_active_pairs(kern, dev);
    if (s2 > 0) slots = s2;
  }
  p.tiles = wide ? wide_tiles : p.m_pairs * ((sh.N + 255) / 256);
  e = ensure_smem_limit(kern, static_cast<int>(GSMEM));
  if (e != cudaSuccess) return e;
  // Persistent: as many CTA pairs as can be resident at once, capped by the
  // number of tiles.
  const int pairs = std::max(1, std::min(p.tiles, slots));
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
  cfg.blockDim = dim3(GTHREADS);
  cfg.dynamicSmemBytes = GSMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&ta, &tb, &tc, &p};
  e = cudaLaunchKernelExC(&cfg, kern, args);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

namespace {

// s: INT4 group scales (kBits = 4, else unused); scale: INT8 per-projection
// scales (kBits = 8, else unused).
template <int kBits>
cudaError_t launch_prefill(const __half* x, const uint32_t* const w[3], const __half* const s[3],
                           const float* scale, __half* const out[3], int M, int N, int K,
                           int num_sms, cudaStream_t stream) {
  using F = PFmt<kBits>;
  CUtensorMap tx, tw[3], ts[3];
  CUresult r = encode_tensor_map_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, x, K, M,
                                    static_cast<uint64_t>(K) * 2, PBK, PBM,
                                    CU_TENSOR_MAP_SWIZZLE_128B);
  if (r != CUDA_SUCCESS) return map_error(r);
  for (int q = 0; q < 3; ++q) {
    r = encode_tensor_map_2d(&tw[q], CU_TENSOR_MAP_DATA_TYPE_UINT32, w[q], N, K * kBits / 32,
                             static_cast<uint64_t>(N) * 4, PBN, F::kRows, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (r != CUDA_SUCCESS) return map_error(r);
    if (kBits == 4) {
      r = encode_tensor_map_2d(&ts[q], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, s[q], N, K / 128,
                               static_cast<uint64_t>(N) * 2, PBN, 1, CU_TENSOR_MAP_SWIZZLE_NONE);
      if (r != CUDA_SUCCESS) return map_error(r);
    } else {
      ts[q] = tx;   // not read by the INT8 kernel
    }
  }
  PrefillParams p{};
  for (int q = 0; q < 3; ++q) {
    p.out[q] = out[q];
    p.scale[q] = kBits == 8 ? scale[q] : 1.f;
  }
  p.M = M;
  p.N = N;
  p.K = K;
  p.m_blocks = (M + PBM - 1) / PBM;
  const int n_blocks = (N + PBN - 1) / PBN;
  p.tiles = p.m_blocks * n_blocks;
  const int grid = std::min(p.tiles, num_sms);
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(tc_qkv_prefill_kernel<kBits>),
                                    static_cast<int>(F::kSmem));
  if (e != cudaSuccess) return e;
  tc_qkv_prefill_kernel<kBits><<<grid, PTHREADS, F::kSmem, stream>>>(tx, tw[0], tw[1], tw[2], ts[0], ts[1],
                                                                     ts[2], p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_w4a16(const __half* x, const uint32_t* const w[3], const __half* const s[3],
                            __half* const out[3], int M, int N, int K, int num_sms,
                            cudaStream_t stream) {
  return launch_prefill<4>(x, w, s, nullptr, out, M, N, K, num_sms, stream);
}

cudaError_t launch_tc_w8a16(const __half* x, const uint32_t* const w[3], const float scale[3],
                            __half* const out[3], int M, int N, int K, int num_sms,
                            cudaStream_t stream) {
  const __half* none[3] = {nullptr, nullptr, nullptr};
  return launch_prefill<8>(x, w, none, scale, out, M, N, K, num_sms, stream);
}

cudaError_t launch_dequant_debug(const uint32_t* w, const __half* s, __half* out, int K, int N,
                                 int variant, cudaStream_t stream) {
  const long long total = static_cast<long long>(K / 8) * N;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks = (total + threads - 1) / threads;
  dequant_debug_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(w, s, out, K, N, variant);
  return cudaGetLastError();
}

unsigned read_and_clear_tc_errors() {
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_tc_err, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
  const unsigned zero = 0;
  cudaMemcpyToSymbol(g_tc_err, &zero, sizeof(zero));
  return v;
}

}  // namespace kaio
