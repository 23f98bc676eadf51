// W4A16 fused QKV projection for decode-sized M (1..16) on the 5th-generation
// tensor cores, split over K across the CTAs of a thread-block cluster.
//
// What it computes ("kaio-candle -- src/qkv_project_int4.rs", doc comment of
// qkv_project_int4): out_p[m, n] = f16(sum_k x[m, k] * RN_f16(int4(W_p[k, n]) *
// s_p[k/128, n])), f32 accumulation, f32 -> f16 in-kernel.
//
// The legacy mma.sync path runs at about a tenth of the tcgen05 rate on this
// GPU, which is below what M = 16 needs to keep up with HBM. Here the product is
// taken transposed, D_p[n, m] = Wd_p^T x^T, on tcgen05 with M = 128 output
// columns (TMEM lanes), N = 16 padded batch rows and K = 16 per instruction:
// * a producer warp streams, per K group of 128 rows, the 16 x 128 packed words
//   and the scale row of each projection plus two 64-wide 128B-swizzled x boxes
//   (rows >= M are zero-filled by TMA) into a ring of shared-memory stages;
// * eight dequant warps (thread = output column = TMEM lane) turn packed
//   words into f16 operands in registers and store them into TMEM A stages;
//   they also permute the staged x chunks to the K order of those operands;
// * three MMA warps, one per projection, issue tcgen05.mma (A from TMEM,
//   B = x tile from shared memory) into that projection's f32 accumulator: at
//   N = 16 the per-instruction issue cost of one warp would leave the tensor
//   core idle most of the time, and three issuers overlap it;
// * the CTAs of a cluster cover consecutive K ranges of the same 128 columns;
//   their accumulators are reduced through distributed shared memory, in rank
//   order (deterministic), and written as f16.
// The kernel takes all 512 TMEM columns; its shared memory keeps it alone on an
// SM, so no CTA ever waits for TMEM. Every
// mbarrier wait is bounded, and both cluster barriers are reached by every
// thread whatever happens.
#include <cuda.h>
#include <cuda_fp16.h>

#include <map>
#include <mutex>
#include <utility>

#include "kaio_device.cuh"
#include "kaio_internal.h"

namespace kaio {

__device__ unsigned g_td_err = 0;

namespace {

constexpr int DN = 128;                  // output columns per CTA (TMEM lanes, MMA M)
constexpr int DM = 16;                   // padded batch rows (MMA N)
constexpr int DGPS = 2;                          // K groups (of 128 K) per shared-memory stage
constexpr int DXBOX = DM * 64 * 2;               // one 64-K x box, 16 rows, 128B-swizzled: 2 KB
constexpr int DX_STAGE = DGPS * 2 * DXBOX;       // 8 KB
constexpr int DMAX_STAGES = 4;
constexpr int DMAX_X = 8;                        // INT8: x ring slots (one stage's x boxes each)

// Two-instruction exact INT4 conversion, for scales 0 < s <= 65504 * 2^-20
// (f16 bits 0x0001 .. 0x2BFF). With nibble pair j moved to bits 4..7 of each
// f16 half, (w & 0x00F000F0) ^ 0x00800080 is the subnormal u * 2^-20 with
// u = n + 8 (the sign bit flipped, as in the general routine), and
// fma(u * 2^-20, s * 2^20, -8 s) rounds the exact value n * s once: it equals
// RN_f16(n * s) bit for bit. s * 2^20 and -8 s are exact in f16 over that
// range. s = 0 or s < 0 would give +0 where n * s is -0 for n <= 0 and is
// left to the general routine, as are larger, infinite and NaN scales.
constexpr uint32_t kFastMask = 0x00F000F0u, kFastMagic = 0x00800080u;
__device__ __forceinline__ uint32_t hfma2_rn(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ bool fast_scale(uint16_t sb) { return static_cast<uint32_t>(sb) - 1u < 0x2BFFu; }
// s * 2^20 (two exact scalings by 1024.0) and -8 s, from s2 = {s, s}
__device__ __forceinline__ void fast_consts(uint32_t s2, uint32_t& sh, uint32_t& sm8) {
  sh = hmul2_rn(hmul2_rn(s2, 0x64006400u), 0x64006400u);
  sm8 = hmul2_rn(s2, 0xC800C800u);
}
// Pair j (nibbles j and j + 4, the order of PairedNibbles) of packed word w.
__device__ __forceinline__ uint32_t fast_pair(uint32_t w, int j, uint32_t sh, uint32_t sm8) {
  const uint32_t src = j == 0 ? w << 4 : (j == 1 ? w : (j == 2 ? w >> 4 : w >> 8));   // pair j at bits 4..7
  return hfma2_rn(and_xor<kFastMask>(src, kFastMagic), sh, sm8);
}
constexpr int DSCALE_ROW = 3 * DN * 2;           // the three scale rows of one K group: 768 B
constexpr int DDQ_WARPS = 8;                     // 2 per TMEM lane quadrant
constexpr int DMMA_WARPS = 3;                    // one per projection
constexpr int DTHREADS = (1 + DMMA_WARPS + DDQ_WARPS) * 32;   // 384
constexpr int DASTAGES = 2;                      // TMEM A stages of one K group (128 K)
constexpr uint32_t DTMEM_COLS = 512;
constexpr uint32_t DA_COL0 = 64;                 // accumulators D[q] at 0..47, A stages after
constexpr uint32_t DA_STAGE_COLS = 192;          // 3 projections x 64 columns (128 K)
constexpr int DRED_BYTES = 3 * DM * DN * 4;      // one CTA's partial tile (24 KB)
constexpr int DSMEM_LIMIT = 232448 - 1024;       // opt-in per-block limit minus static shared memory
constexpr size_t DSMEM = DSMEM_LIMIT;
static_assert(DA_COL0 + DASTAGES * DA_STAGE_COLS <= DTMEM_COLS, "TMEM layout");

// Stage layout of one weight format (kBits = 4: INT4 with f16 group scales;
// kBits = 8: INT8 with one f32 scale per projection, applied in the epilogue).
//
// INT8 keeps its x boxes in a ring of their own (kSplitX): a weight stage is
// refilled as soon as its words are in the conversion warps' registers, while
// the x boxes stay until the MMAs reading them are done. Its 96 KB weight
// stages are few (two fit), and this freed them ~10 % sooner at M = 16,
// K = N = 8192 (38.4 -> 35.0 us). INT4 (48 KB of words per stage, x permuted
// in place by the dequant warps) measured slower that way (30.1 -> 32.4 us)
// and keeps x and words in one stage.
template <int kBits>
struct DFmt {
  static constexpr bool kSplitX = kBits == 8;
  static constexpr int kRows = 128 * kBits / 32;        // packed rows per K group: 16 or 32
  static constexpr int kWBox = DGPS * kRows * DN * 4;   // one projection's words per stage: 16 or 32 KB
  static constexpr int kXIn = kSplitX ? 0 : DX_STAGE;   // x bytes inside a stage (before the words)
  static constexpr int kStage = kXIn + 3 * kWBox;       // 56 KB (x + words) or 96 KB (words)
  static_assert(kStage % 1024 == 0, "x boxes stay 1024-aligned");
  static_assert(DRED_BYTES <= kStage, "partials reuse the ring");
};

struct DecTcParams {
  __half* out[3];
  float scale[3];  // INT8: per-projection scales
  int M, N, K;
  int tiles;     // ceil(N / 128) column tiles (each covers Q, K and V)
  int S;         // cluster size: K ranges per column tile
  int ng;        // K / 128
  int nst;       // ring stages (DGPS K groups each)
  int nx;        // INT8: x ring slots (one stage's x boxes each)
  int x_off;     // INT8: byte offset of the x ring (after the stage ring)
  int s_off;     // byte offset of the scale rows (after the rings)
  int sbox;      // scale rows per TMA box
  unsigned long long wait_ns;   // limit of every pipeline wait (kWaitLimitNs; shorter in a test)
};

template <int kBits>
__global__ void __launch_bounds__(DTHREADS, 1)
    tc_decode_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW0,
                     const __grid_constant__ CUtensorMap tmW1, const __grid_constant__ CUtensorMap tmW2,
                     const __grid_constant__ CUtensorMap tmS0, const __grid_constant__ CUtensorMap tmS1,
                     const __grid_constant__ CUtensorMap tmS2, const DecTcParams p) {
  using F = DFmt<kBits>;
  constexpr int DW_BOX = F::kWBox, DSTAGE_BYTES = F::kStage;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = align_smem_1024(smem_raw);
  __shared__ __align__(8) uint64_t full[DMAX_STAGES], empty[DMAX_STAGES], xfull[DMAX_X], xempty[DMAX_X], sbar0,
      sbar, a_full[DASTAGES], a_empty[DASTAGES], acc_full, mma_done[DMMA_WARPS];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_ctarank());
  const int tile = blockIdx.x / p.S;
  const int n0 = tile * DN;
  const int g_begin = rank * p.ng / p.S;
  const int nsg = (rank + 1) * p.ng / p.S - g_begin;     // K groups of this CTA
  const int nstg = (nsg + DGPS - 1) / DGPS;              // shared-memory stages of this CTA
  volatile int* abort = &abort_flag;

  // Producer state (thread 0). The first copies are issued before the TMEM
  // allocation and the block barrier so that their latency overlaps the
  // set-up, in the order the consumers need them: stage 0, the first box of
  // scale rows, stage 1, the other scale boxes; the rest of the ring follows
  // once stage 0 has landed (every SM asks for its first stages at the same
  // moment, and copies issued together land together).
  uint32_t fills[DMAX_STAGES] = {0, 0, 0, 0};
  uint32_t xfills[DMAX_X] = {};
  int pst = 0, pi = 0, xi = 0;
  uint32_t pph = 0;
  const int nsb = kBits == 4 ? (nsg + p.sbox - 1) / p.sbox : 0;   // boxes of scale rows
  auto issue_stage = [&]() {
    unsigned char* sx = smem + pst * DSTAGE_BYTES;
    unsigned char* sw = sx + F::kXIn;
    const int g = g_begin + pi * DGPS;
    mbar_arrive_expect_tx(&full[pst], DSTAGE_BYTES);
    tma_load_2d(sw, &tmW0, &full[pst], n0, g * F::kRows);
    tma_load_2d(sw + DW_BOX, &tmW1, &full[pst], n0, g * F::kRows);
    tma_load_2d(sw + 2 * DW_BOX, &tmW2, &full[pst], n0, g * F::kRows);
    if constexpr (!F::kSplitX) {
#pragma unroll
      for (int b = 0; b < 2 * DGPS; ++b)
        tma_load_2d(sx + b * DXBOX, &tmX, &full[pst], (g * 2 + b) * 64, 0);
    }
    ++fills[pst];
    ++pi;
    if (++pst == p.nst) { pst = 0; pph ^= 1; }
  };
  auto issue_x = [&]() {                          // INT8: stage xi's x boxes into the x ring
    const int xs = xi % p.nx;
    unsigned char* sx = smem + p.x_off + xs * DX_STAGE;
    const int g = g_begin + xi * DGPS;
    mbar_arrive_expect_tx(&xfull[xs], DX_STAGE);
#pragma unroll
    for (int b = 0; b < 2 * DGPS; ++b)
      tma_load_2d(sx + b * DXBOX, &tmX, &xfull[xs], (g * 2 + b) * 64, 0);
    ++xfills[xs];
    ++xi;
  };
  auto issue_scales = [&](int b, uint64_t* bar) {
    unsigned char* ss = smem + p.s_off + b * p.sbox * DSCALE_ROW;
    tma_load_2d(ss, &tmS0, bar, n0, g_begin + b * p.sbox);
    tma_load_2d(ss + p.sbox * DN * 2, &tmS1, bar, n0, g_begin + b * p.sbox);
    tma_load_2d(ss + 2 * p.sbox * DN * 2, &tmS2, bar, n0, g_begin + b * p.sbox);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.nst; ++s) {
      mbar_init(&full[s], 1);
      // dequant warps (+ one commit per MMA warp when the stage holds x)
      mbar_init(&empty[s], DDQ_WARPS + (F::kSplitX ? 0 : DMMA_WARPS));
    }
    if constexpr (F::kSplitX) {
      for (int s = 0; s < p.nx; ++s) {
        mbar_init(&xfull[s], 1);
        mbar_init(&xempty[s], DMMA_WARPS);            // one commit per MMA warp
      }
    }
    mbar_init(&sbar0, 1);
    mbar_init(&sbar, 1);
    for (int a = 0; a < DASTAGES; ++a) {
      mbar_init(&a_full[a], DDQ_WARPS / 2);       // the set of dequant warps owning stage a
      mbar_init(&a_empty[a], DMMA_WARPS);
    }
    mbar_init(&acc_full, DMMA_WARPS);
    for (int w = 0; w < DMMA_WARPS; ++w) mbar_init(&mma_done[w], 1);
    abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW0); tma_prefetch_desc(&tmW1); tma_prefetch_desc(&tmW2);
    if (kBits == 4) {
      tma_prefetch_desc(&tmS0); tma_prefetch_desc(&tmS1); tma_prefetch_desc(&tmS2);
    }
    // While the preceding kernel finishes, start pulling the weights of this
    // CTA's first stage from HBM into L2 (hints only, see tma_prefetch_l2_2d),
    // so that its copies after the wait find them there. Only the first stage:
    // prefetching a CTA's whole range evicts lines before use on workloads
    // near the L2 size, and deeper L2 look-ahead of the ring slowed M = 1.
    if (nstg > 0) {
      tma_prefetch_l2_2d(&tmW0, n0, g_begin * F::kRows);
      tma_prefetch_l2_2d(&tmW1, n0, g_begin * F::kRows);
      tma_prefetch_l2_2d(&tmW2, n0, g_begin * F::kRows);
    }
    grid_dependency_wait();                       // the previous kernel's writes are visible
    if (nstg > 0) {
      issue_stage();
      if constexpr (F::kSplitX) issue_x();
    }
    if (nsb > 0) {
      mbar_arrive_expect_tx(&sbar0, static_cast<uint32_t>(3 * p.sbox * DN * 2));
      issue_scales(0, &sbar0);
    }
    if (pi < nstg && pi < p.nst) {
      issue_stage();
      if constexpr (F::kSplitX) issue_x();
    }
    if (nsb > 1) {
      mbar_arrive_expect_tx(&sbar, static_cast<uint32_t>(3 * (nsb - 1) * p.sbox * DN * 2));
      for (int b = 1; b < nsb; ++b) issue_scales(b, &sbar);
    }
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base_sh, DTMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  grid_dependency_wait();                         // returns at once: thread 0 has waited
  allow_dependents_launch();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Few, large copies: per stage one 16 KB box of packed words per projection
    // and four 2 KB x boxes; the scale rows of the whole K range (issued above
    // with the first two stages).
    if (lane == 0) {
      bool ok = pi >= nstg || pi >= p.nst || mbar_wait_lim(&full[0], 0, abort, &g_td_err, p.wait_ns);
      while (ok && pi < nstg && pi < p.nst) issue_stage();   // the rest of the first ring(s)
      if constexpr (F::kSplitX)
        while (ok && xi < nstg && xi < p.nx) issue_x();
      while (ok && pi < nstg) {
        if (!mbar_wait_lim(&empty[pst], pph ^ 1, abort, &g_td_err, p.wait_ns)) break;
        issue_stage();
        if constexpr (F::kSplitX) {
          // x of stage xi reuses the slot of stage xi - nx (nx >= nst: its
          // MMAs finished long before)
          while (ok && xi < pi && xi < nstg) {
            if (!mbar_wait_lim(&xempty[xi % p.nx], ((xi / p.nx) - 1) & 1, abort, &g_td_err, p.wait_ns)) {
              ok = false;
              break;
            }
            issue_x();
          }
        }
      }
      if constexpr (F::kSplitX) {
        while (ok && xi < nstg) {
          if (!mbar_wait_lim(&xempty[xi % p.nx], ((xi / p.nx) - 1) & 1, abort, &g_td_err, p.wait_ns)) break;
          issue_x();
        }
        for (int s2 = 0; s2 < p.nx; ++s2)
          if (xfills[s2]) mbar_wait_drain(&xfull[s2], (xfills[s2] - 1) & 1, &g_td_err);
      }
      for (int s2 = 0; s2 < p.nst; ++s2)
        if (fills[s2]) mbar_wait_drain(&full[s2], (fills[s2] - 1) & 1, &g_td_err);
      if (nsb > 0) mbar_wait_drain(&sbar0, 0, &g_td_err);
      if (nsb > 1) mbar_wait_drain(&sbar, 0, &g_td_err);
    }
  } else if (warp <= DMMA_WARPS) {
    // ------------------------------------------------------------ MMA warps
    // MMA warp q issues the eight 16-K steps of every K group of projection q
    // into that projection's accumulator D[q]. At N = 16 the per-instruction
    // issue cost dominates; three issuing warps overlap it. A group's A stage
    // being full implies its x boxes have landed and been permuted (the
    // dequant warps do both before their hand-off), so these warps wait on
    // nothing else.
    const int q = warp - 1;
    const uint32_t dq = tmem + static_cast<uint32_t>(q * DM);
    constexpr uint32_t idesc = idesc_f16_f32(DN, DM, false, false);
    int a = 0, st = 0;
    uint32_t aph = 0;
    bool ok = true;
    for (int i = 0; i < nstg && ok; ++i) {
      const int xs = i % p.nx;
      unsigned char* sx = F::kSplitX ? smem + p.x_off + xs * DX_STAGE : smem + st * DSTAGE_BYTES;
      const uint64_t bd0 = sdesc_sw128(smem_u32(sx), 16, 1024);
      const uint32_t blo = static_cast<uint32_t>(bd0), bhi = static_cast<uint32_t>(bd0 >> 32);
      const int ngs = min(DGPS, nsg - i * DGPS);
      for (int j = 0; j < ngs; ++j) {              // K groups of this stage
        if (!mbar_wait_lim(&a_full[a], aph, abort, &g_td_err, p.wait_ns)) { ok = false; break; }
        if (lane == 0) {
          tc_fence_after();
          const uint32_t acc0 = (i | j) != 0 ? 1u : 0u;
          const uint32_t abase = tmem + DA_COL0 + static_cast<uint32_t>(a * DA_STAGE_COLS + q * 64);
          const uint32_t xlo = blo + static_cast<uint32_t>((2 * j * DXBOX) >> 4);
          // MMA step (hh, kk) covers K 64hh + 16kk .. +15 of the group: x box hh,
          // chunk kk; its A columns are kk*16 + hh*8 (INT4: the dequant warps'
          // interleaved order) or 32hh + 8kk (INT8: K pairs in order).
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_ts_lohi(dq, abase + (kBits == 4 ? kk * 16 + hh * 8 : hh * 32 + kk * 8),
                           xlo + ((hh * DXBOX + kk * 32) >> 4), bhi, idesc, (hh | kk) != 0 ? 1u : acc0);
          umma_commit(&a_empty[a]);
          if (j == ngs - 1) umma_commit(F::kSplitX ? &xempty[xs] : &empty[st]);
        }
        __syncwarp();
        if (++a == DASTAGES) { a = 0; aph ^= 1; }
      }
      if (++st == p.nst) st = 0;
    }
    if (lane == 0) {
      if (ok) umma_commit(&acc_full);              // fires when this warp's MMAs are done
      umma_commit(&mma_done[q]);
      mbar_wait_drain(&mma_done[q], 0, &g_td_err);
    }
  } else {
    // ------------------------------------------------------------ dequant warps
    // Two sets of four warps (one per TMEM lane quadrant). Set js takes the
    // K groups with j == js in every shared-memory stage (even / odd groups)
    // and owns TMEM A stage js, so each set waits only for the MMAs of its
    // own previous group: the sets drift out of phase and one set's waits and
    // loads overlap the other set's arithmetic. Thread = output column
    // n0 + 32*sp + lane = TMEM lane; it dequantises all 16 packed rows of its
    // column for the three projections (48 words per group).
    const int sp = warp & 3;
    const int js = (warp - 1 - DMMA_WARPS) >> 2;
    const int nl = 32 * sp + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * sp) << 16;
    const unsigned char* scale_base = smem + p.s_off + nl * 2;
    int st = 0;
    uint32_t aph = 0, ph = 0;
    bool ok = nsb == 0 || mbar_wait_lim(&sbar0, 0, abort, &g_td_err, p.wait_ns);
    bool have_scales = nsb <= 1;                 // rows of the later scale boxes have landed
    // x chunks this thread permutes in its groups: the two 64-K boxes 2js and
    // 2js+1 of a group hold 2 x 16 rows x 8 chunks = 256 chunks, two per
    // thread of the set (rows >= M are zeros and stay so).
    const int pt = (threadIdx.x - (1 + DMMA_WARPS) * 32) & 127;
    const int pm = (pt >> 3) & 15, pc = pt & 7;
    const int poff = 2 * js * DXBOX + (pm >> 3) * 1024 + (pm & 7) * 128 + ((pc ^ (pm & 7)) << 4);
    const uint32_t tbase = tmem + lane_base + DA_COL0 + js * DA_STAGE_COLS;
    for (int i = 0; i < nstg && ok; ++i) {
      const int ngs = min(DGPS, nsg - i * DGPS);
      if (js < ngs) {
        if (!mbar_wait_lim(&full[st], ph, abort, &g_td_err, p.wait_ns)) { ok = false; break; }
        if (kBits == 4 && pm < p.M) {
          permute_x_chunk(smem + st * DSTAGE_BYTES + poff);
          permute_x_chunk(smem + st * DSTAGE_BYTES + poff + DXBOX);
          fence_proxy_async_smem();               // the MMAs read x through the async proxy
        }
        if constexpr (kBits == 8) {
          // The stage's x boxes (own ring) have landed before this set hands
          // its A stage to the MMAs that read them.
          if (!mbar_wait_lim(&xfull[i % p.nx], static_cast<uint32_t>(i / p.nx) & 1u, abort, &g_td_err,
                             p.wait_ns)) {
            ok = false;
            break;
          }
          // Thread = column nl: its 32 packed rows of the group per projection,
          // converted exactly to f16 K pairs. Column c of projection q's 64 holds
          // K pair c (K-rows 2c, 2c+1: byte pair c % 2 of packed row c / 2).
          if (!mbar_wait_lim(&a_empty[js], aph ^ 1, abort, &g_td_err, p.wait_ns)) { ok = false; break; }
          tc_fence_after();
          const uint32_t* sw = reinterpret_cast<const uint32_t*>(smem + st * DSTAGE_BYTES + F::kXIn) +
                               js * F::kRows * DN + nl;
#pragma unroll
          for (int q = 0; q < 3; ++q)
#pragma unroll
            for (int k2 = 0; k2 < 2; ++k2) {
              uint32_t v[32];
#pragma unroll
              for (int rr = 0; rr < 16; ++rr)
                int8x4_to_half2x2(sw[q * (DW_BOX / 4) + (k2 * 16 + rr) * DN], v[2 * rr], v[2 * rr + 1]);
              tmem_st32(tbase + q * 64 + k2 * 32, v);
            }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[st]);   // this set's words of the stage have been read
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&a_full[js]);
          aph ^= 1;
          if (++st == p.nst) { st = 0; ph ^= 1; }
          continue;
        }
        const int gl = i * DGPS + js;             // group index inside the CTA's range
        if (!have_scales && gl >= p.sbox) {
          if (!mbar_wait_lim(&sbar, 0, abort, &g_td_err, p.wait_ns)) { ok = false; break; }
          have_scales = true;
        }
        // scale rows of group gl: box gl/8 (boxes hold up to 8 rows), row gl%8
        const unsigned char* sc = scale_base + (gl >> 3) * p.sbox * DSCALE_ROW + (gl & 7) * (DN * 2);
        const unsigned char* sw = smem + st * DSTAGE_BYTES + F::kXIn + js * 16 * (DN * 4) + nl * 4;
        uint32_t wd[3][16], s2[3];                // wd[q][row]: packed rows 0..15 of the group
        bool small = true;                        // all three scales in the two-instruction range
#pragma unroll
        for (int q = 0; q < 3; ++q) {
          const uint16_t sb = *reinterpret_cast<const uint16_t*>(sc + q * p.sbox * DN * 2);
          s2[q] = half2_bits(sb, sb);
          small = small && fast_scale(sb);
#pragma unroll
          for (int r = 0; r < 16; ++r)
            wd[q][r] = *reinterpret_cast<const uint32_t*>(sw + q * DW_BOX + r * (DN * 4));
        }
        const bool fast = __all_sync(0xffffffffu, small);   // the warp takes one routine
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);   // this set's words of the stage are in registers
        if (!mbar_wait_lim(&a_empty[js], aph ^ 1, abort, &g_td_err, p.wait_ns)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < 3; ++q)
#pragma unroll
          for (int k2 = 0; k2 < 2; ++k2) {
            // column kk*16 + hh*8 + 4*rr + jj (kk = 2*k2 + kx) of projection q's 64
            // holds K pair jj of packed row hh*8 + 2*kk + rr (the A layout of an MMA
            // step); one 32-column store covers MMA steps 2*k2 and 2*k2+1
            uint32_t v[32];
            if (fast) {
              uint32_t sh, sm8;
              fast_consts(s2[q], sh, sm8);
              // in two passes (the 32 LOP3, then the 32 FMAs), so that each warp
              // has independent instructions to issue while results are in
              // flight: two dequant warps per scheduler hide little latency
              // (M=16, K=N=8192: 29.35 -> 29.11 us)
#pragma unroll
              for (int kx = 0; kx < 2; ++kx)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                  for (int rr = 0; rr < 2; ++rr) {
                    const uint32_t w = wd[q][hh * 8 + 2 * (2 * k2 + kx) + rr];
                    const uint32_t src[4] = {w << 4, w, w >> 4, w >> 8};   // pair j at bits 4..7
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                      v[kx * 16 + hh * 8 + 4 * rr + jj] = and_xor<kFastMask>(src[jj], kFastMagic);
                  }
#pragma unroll
              for (int c = 0; c < 32; ++c) asm volatile("" : "+r"(v[c]));   // keep the passes apart
#pragma unroll
              for (int c = 0; c < 32; ++c) v[c] = hfma2_rn(v[c], sh, sm8);
            } else {
#pragma unroll
              for (int kx = 0; kx < 2; ++kx)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                  for (int rr = 0; rr < 2; ++rr) {
                    const PairedNibbles pn(wd[q][hh * 8 + 2 * (2 * k2 + kx) + rr]);
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) v[kx * 16 + hh * 8 + 4 * rr + jj] = pn.pair(jj, s2[q]);
                  }
            }
            tmem_st32(tbase + q * 64 + k2 * 32, v);
          }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[js]);
        aph ^= 1;
      } else {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);   // no group of this set in the CTA's last stage
      }
      if (++st == p.nst) { st = 0; ph ^= 1; }
    }

    // Epilogue part 1: this CTA's partial D[q][n][m] -> shared
    // red[q][m][n] (set js drains batch rows 8js .. 8js+7). The ring is free
    // once every MMA has completed (acc_full).
    float* red = reinterpret_cast<float*>(smem);
    const bool have = ok && nsg > 0 && mbar_wait_lim(&acc_full, 0, abort, &g_td_err, p.wait_ns);
    if (have) tc_fence_after();
    uint32_t r[3][8];
    if (have) {
#pragma unroll
      for (int q = 0; q < 3; ++q) tmem_ld8(tmem + lane_base + q * DM + js * 8, r[q]);
      tmem_ld_wait();
    }
#pragma unroll
    for (int q = 0; q < 3; ++q)
#pragma unroll
      for (int jj = 0; jj < 8; ++jj)
        red[(q * DM + js * 8 + jj) * DN + nl] = have ? __uint_as_float(r[q][jj]) : 0.f;
    tc_fence_before();
  }

  // Epilogue part 2: rank r finishes batch rows m with m % S == r, summing the
  // S partials in rank order through distributed shared memory, four columns
  // at a time.
  __syncwarp();
  cluster_sync_all();
  {
    const int dt = threadIdx.x;
    const uint32_t red_s = smem_u32(smem);
    const int rows = (p.M - rank + p.S - 1) / p.S;      // rows rank, rank+S, ... below M
    const int items = rows * 3 * (DN / 4);
    for (int it = dt; it < items; it += DTHREADS) {
      const int m = rank + (it / (3 * (DN / 4))) * p.S;
      const int q = (it / (DN / 4)) % 3;
      const int n4 = it % (DN / 4);
      const uint32_t off = static_cast<uint32_t>(((q * DM + m) * DN + 4 * n4) * 4);
      float4 v[8];
#pragma unroll
      for (int r = 0; r < 8; ++r)
        if (r < p.S) v[r] = dsmem_ld_f4(dsmem_map(red_s + off, static_cast<uint32_t>(r)));
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int r = 0; r < 8; ++r)
        if (r < p.S) {
          acc.x += v[r].x; acc.y += v[r].y; acc.z += v[r].z; acc.w += v[r].w;
        }
      if (kBits == 8) {
        const float sc = q == 0 ? p.scale[0] : (q == 1 ? p.scale[1] : p.scale[2]);
        acc.x *= sc; acc.y *= sc; acc.z *= sc; acc.w *= sc;
      }
      const int c4 = n0 + 4 * n4;
      if (c4 < p.N) {
        __half* out = q == 0 ? p.out[0] : (q == 1 ? p.out[1] : p.out[2]);
        const __half2 lo = __floats2half2_rn(acc.x, acc.y);
        const __half2 hi = __floats2half2_rn(acc.z, acc.w);
        uint2 u;
        u.x = *reinterpret_cast<const uint32_t*>(&lo);
        u.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(out + static_cast<size_t>(m) * p.N + c4) = u;
      }
    }
  }
  __syncwarp();
  cluster_sync_all();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, DTMEM_COLS);
  }
}

template <int kBits>
int dec_max_active_clusters(int S, int dev) {
  static std::mutex mu;
  static std::map<std::pair<int, int>, int> cache;
  std::lock_guard<std::mutex> lk(mu);
  const auto key = std::make_pair(dev, S);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int n = 0;
  const void* kern = reinterpret_cast<const void*>(tc_decode_kernel<kBits>);
  if (ensure_smem_limit(kern, static_cast<int>(DSMEM)) == cudaSuccess) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(S * 64));
    cfg.blockDim = dim3(DTHREADS);
    cfg.dynamicSmemBytes = 120 * 1024;
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

template <int kBits>
TcDecodePlan plan_dec(int M, int N, int K, int dev) {
  TcDecodePlan pl{};
  pl.tiles = (N + DN - 1) / DN;
  pl.ng = K / 128;
  double best = -1;
  for (int S = 1; S <= 8 && S <= pl.ng; ++S) {
    const int range = (pl.ng + S - 1) / S;
    const int sbytes = kBits == 4 ? ((range + 7) / 8) * 8 * DSCALE_ROW : 0;
    // scales + 2 stages (+ 2 x slots) must fit
    if (sbytes + 2 * (DFmt<kBits>::kStage + DX_STAGE - DFmt<kBits>::kXIn) + 2048 > DSMEM_LIMIT) continue;
    const int slots = dec_max_active_clusters<kBits>(S, dev);
    if (slots <= 0) continue;
    const long long waves = (pl.tiles + slots - 1) / slots;
    // Cost: K groups the busiest SM streams, plus a fixed start-up cost per wave.
    const double est = static_cast<double>(waves) * (range + 2.0);
    if (best < 0 || est < best - 1e-9) {
      best = est;
      pl.S = S;
    }
  }
  pl.ok = best > 0 && M <= DM;
  return pl;
}

// s: INT4 group scales (kBits = 4, else unused); scale: INT8 per-projection
// scales (kBits = 8, else unused).
template <int kBits>
cudaError_t launch_dec(const __half* x, const uint32_t* const w[3], const __half* const s[3],
                       const float* scale, __half* const out[3], int M, int N, int K,
                       const TcDecodePlan& pl, cudaStream_t stream,
                       unsigned long long wait_ns = kWaitLimitNs) {
  using F = DFmt<kBits>;
  const int range = (pl.ng + pl.S - 1) / pl.S;
  const int sbox = kBits == 4 ? std::min(8, pl.ng) : 1;
  const int sbytes = kBits == 4 ? ((range + sbox - 1) / sbox) * sbox * DSCALE_ROW : 0;
  DecTcParams p{};
  for (int q = 0; q < 3; ++q) {
    p.out[q] = out[q];
    p.scale[q] = kBits == 8 ? scale[q] : 1.f;
  }
  p.M = M;
  p.N = N;
  p.K = K;
  p.tiles = pl.tiles;
  p.S = pl.S;
  p.ng = pl.ng;
  p.sbox = sbox;
  p.wait_ns = wait_ns;
  const int nstg = (range + DGPS - 1) / DGPS;
  if constexpr (F::kSplitX) {
    // as many stages as fit (up to DMAX_STAGES) with an x ring twice as deep
    // (up to DMAX_X, never more than the CTA's stages)
    p.nst = 1;
    p.nx = std::min(nstg, 2);
    for (int ns = std::min(nstg, DMAX_STAGES); ns >= 1; --ns) {
      const int nx = std::max(1, std::min(nstg, std::min(DMAX_X, 2 * ns)));
      if (ns * F::kStage + nx * DX_STAGE + sbytes + 1024 <= DSMEM_LIMIT) {
        p.nst = ns;
        p.nx = nx;
        break;
      }
    }
  } else {
    p.nst = std::min(std::min(nstg, DMAX_STAGES), (DSMEM_LIMIT - 1024 - sbytes) / F::kStage);
    p.nst = std::max(p.nst, 1);
    p.nx = 1;                                     // x travels inside the stages
  }
  p.x_off = p.nst * F::kStage;
  p.s_off = p.x_off + (F::kSplitX ? p.nx * DX_STAGE : 0);
  const size_t smem_used = static_cast<size_t>(p.s_off + sbytes + 1024);
  CUtensorMap tx, tw[3], ts[3];
  CUresult r = encode_tensor_map_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, x, K, M,
                                    static_cast<uint64_t>(K) * 2, 64, DM, CU_TENSOR_MAP_SWIZZLE_128B);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  for (int q = 0; q < 3; ++q) {
    r = encode_tensor_map_2d(&tw[q], CU_TENSOR_MAP_DATA_TYPE_UINT32, w[q], N, K * kBits / 32,
                             static_cast<uint64_t>(N) * 4, DN, DGPS * F::kRows, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (kBits == 4) {
      r = encode_tensor_map_2d(&ts[q], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, s[q], N, K / 128,
                               static_cast<uint64_t>(N) * 2, DN, sbox, CU_TENSOR_MAP_SWIZZLE_NONE);
      if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    } else {
      ts[q] = tx;   // not read by the INT8 kernel
    }
  }
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(tc_decode_kernel<kBits>),
                                    static_cast<int>(DSMEM));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(pl.tiles * pl.S));
  cfg.blockDim = dim3(DTHREADS);
  // Always more than half the SM's shared memory: the kernel takes all of TMEM
  // and must be alone on its SM.
  cfg.dynamicSmemBytes = std::max(smem_used, static_cast<size_t>(120 * 1024));
  cfg.stream = stream;
  // Programmatic stream serialization: the next call's CTAs may start (and set
  // up) on free SMs before this one ends; each waits for its predecessor with
  // grid_dependency_wait() before touching global memory.
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(pl.S);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, tc_decode_kernel<kBits>, tx, tw[0], tw[1], tw[2], ts[0], ts[1], ts[2], p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}


// The dequant stage of the decode kernel alone, for bit-exact tests: each
// packed word with the two-instruction routine where its scale allows, the
// paired-nibble routine elsewhere; out[8r + i][n] in K-row order.
__global__ void dequant_fast_debug_kernel(const uint32_t* __restrict__ w, const __half* __restrict__ s,
                                          __half* __restrict__ out, int K, int N) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long total = static_cast<long long>(K / 8) * N;
  if (idx >= total) return;
  const int r = static_cast<int>(idx / N), n = static_cast<int>(idx % N);
  const uint32_t word = w[idx];
  const uint16_t sb = __half_as_ushort(s[static_cast<size_t>(r / 16) * N + n]);
  const uint32_t s2 = half2_bits(sb, sb);
  uint32_t sh, sm8;
  fast_consts(s2, sh, sm8);
  const PairedNibbles pn(word);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t v = fast_scale(sb) ? fast_pair(word, j, sh, sm8) : pn.pair(j, s2);
    out[static_cast<size_t>(8 * r + j) * N + n] = __ushort_as_half(static_cast<uint16_t>(v & 0xFFFFu));
    out[static_cast<size_t>(8 * r + j + 4) * N + n] = __ushort_as_half(static_cast<uint16_t>(v >> 16));
  }
}

}  // namespace

// The plan depends on (device, N, K, M <= 16) only; the last few are kept per
// host thread, so a decode loop does not search cluster shapes on every call.
template <int kBits>
TcDecodePlan plan_dec_cached(int M, int N, int K, int dev) {
  struct Entry {
    int dev, N, K;
    bool small;
    TcDecodePlan pl;
  };
  thread_local Entry recent[8];
  thread_local int n_recent = 0, next = 0;
  const bool small = M <= DM;
  for (int i = 0; i < n_recent; ++i)
    if (recent[i].dev == dev && recent[i].N == N && recent[i].K == K && recent[i].small == small)
      return recent[i].pl;
  const TcDecodePlan pl = plan_dec<kBits>(M, N, K, dev);
  recent[next] = Entry{dev, N, K, small, pl};
  next = (next + 1) % 8;
  if (n_recent < 8) ++n_recent;
  return pl;
}

TcDecodePlan plan_tc_decode(int M, int N, int K, int dev) { return plan_dec_cached<4>(M, N, K, dev); }
TcDecodePlan plan_tc_decode_int8(int M, int N, int K, int dev) { return plan_dec_cached<8>(M, N, K, dev); }

cudaError_t launch_tc_decode(const __half* x, const uint32_t* const w[3], const __half* const s[3],
                             __half* const out[3], int M, int N, int K, const TcDecodePlan& pl,
                             cudaStream_t stream) {
  return launch_dec<4>(x, w, s, nullptr, out, M, N, K, pl, stream);
}

cudaError_t launch_tc_decode_wait_limit(const __half* x, const uint32_t* const w[3], const __half* const s[3],
                                        __half* const out[3], int M, int N, int K, const TcDecodePlan& pl,
                                        unsigned long long wait_ns, cudaStream_t stream) {
  return launch_dec<4>(x, w, s, nullptr, out, M, N, K, pl, stream, wait_ns);
}

cudaError_t launch_tc_decode_int8(const __half* x, const uint32_t* const w[3], const float scale[3],
                                  __half* const out[3], int M, int N, int K, const TcDecodePlan& pl,
                                  cudaStream_t stream) {
  const __half* none[3] = {nullptr, nullptr, nullptr};
  return launch_dec<8>(x, w, none, scale, out, M, N, K, pl, stream);
}

unsigned read_and_clear_tc_decode_errors() {
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_td_err, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
  const unsigned zero = 0;
  cudaMemcpyToSymbol(g_td_err, &zero, sizeof(zero));
  return v;
}

cudaError_t launch_dequant_fast_debug(const uint32_t* w, const __half* s, __half* out, int K, int N,
                                      cudaStream_t stream) {
  const long long total = static_cast<long long>(K / 8) * N;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks = (total + threads - 1) / threads;
  dequant_fast_debug_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(w, s, out, K, N);
  return cudaGetLastError();
}

}  // namespace kaio
