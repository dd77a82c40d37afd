// MXFP8 low-batch GEMM with a publishing epilogue, for sm_103a.
//
// C[t][n] = sum_k W[n][k] x[t][k] (page "vllm.models.deepseek_v41.nvidia.
// specialized_decode.boundary.publishing_gemm", module description "GEMM
// structure"): the weight is the MMA's A operand (128 output columns per CTA,
// N/128 tiles; 128/F when folded, below), the at most 8 activation rows its
// B operand (N = 8).  Each
// CTA of a split-K cluster of S multiplies one K slice; the partials are
// exchanged through distributed shared memory and each CTA reduces 1/S of
// the tokens.  The epilogue rounds to BF16, writes C, and publishes every
// value with negative zero cleared into generation stage_state[0] of the
// mailbox as aligned 16-byte packs of eight consecutive columns, then one
// thread sets stage_state[1] (same page, publish_value and epilog_warp).
//
// Accumulation.  The tensor core's own FP32 accumulation over a long K loses
// too much on outputs that nearly cancel, so partial sums leave tensor memory
// early: each MMA (or each group of acc_blocks MMAs) writes a fresh
// accumulator slot of a ring, and the epilogue warps fold every slot into a
// compensated FP32 pair (hi + lo, Knuth's TwoSum) as soon as it completes.
// The pair is rounded once to BF16 (hi + lo taken exactly, from its FP32
// bits).
//
// Folding (F = 1, 2, 4 or 8).  A grid of N/128 x S CTAs leaves most SMs idle
// on small shapes, and one SM streams at most about 70-120 GB/s.  With F > 1
// a CTA owns 128/F output columns and stacks F consecutive 128-wide K pieces
// of its weight rows in the MMA's 128 rows (rows [p R, (p+1) R) hold piece p,
// R = 128/F), the activations as F groups of 8 columns (N = 8 F, group p =
// piece p), so one stage is still 16 KB of W and 4 MMAs.  Of the 128 x 8F
// product only the F diagonal blocks (rows of piece p, columns of group p)
// are kept; the epilogue adds the F pieces of each output column.  The grid
// has F times more CTAs for the same weight bytes and MMA count.  At F = 8
// (16-row tiles, unsplit only) a warp's 32 lanes span two pieces, while a
// tensor-memory load takes one column address per warp: each warp loads both
// pieces' columns and each lane keeps its own eight.
//
// Warp roles (pipes = 1, 2 or 4 per launch):
//   warp 0      TMA producer: one lane per pipe, lane l taking stages
//               l, l + pipes, ...; per stage the W tile + W scale chunk
//               (started before the programmatic grid wait) and the F x
//               tiles.
//   warp 1, 6.. MMA issuers, one warp per pipe (warp 1 also allocates tensor
//               memory): one thread each issues, per stage, tcgen05.cp of the
//               W and x scale chunks and one block-scaled tcgen05.mma per
//               32-wide K block.  Blocks have 160 + 32 * pipes threads.
//   warps 2-5   epilogue: x scales staged for the copies, partial sums read
//               back (tcgen05.ld 32x32b: thread = MMA row, registers =
//               tokens of its diagonal block) and folded into the compensated
//               sums, the F pieces of a column added, split-K exchange, BF16
//               rounding, C store, publish.
//
// Tensor-memory columns: [acc, +acc_ring * acc_slot) the accumulator ring (FP32,
// lane = MMA row, column = block * 8 F + piece * 8 + token); then the W and x
// scale rings, one 4-column slot per K tile of the shared-memory ring each,
// filled by tcgen05.cp (32x128b, multicast to the four lane quarters) from
// 16-byte-row scale chunks in shared memory.  Every scale address is 4-column
// aligned.
//
// Stages of two K tiles (T = 2, cta_k 256): a stage's two tiles share one
// full and one empty barrier and arrive with one W copy, one W-scale copy and
// one x load; each tile keeps its own accumulator slot and scale slots, so
// the sums run in the same order and the bits match T = 1.
//
// The kernel template lives in this header so its instantiations can be
// spread over translation units that compile in parallel: publish_gemm.cu
// (F = 1) and publish_gemm_fold.cu (F = 2, 4, 8).
#pragma once
#include <cuda_bf16.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace mxfp8 {
namespace {

// The 16x256b load's transpose buffer inside W stage 0: 4 warps x 32 columns
// x 8 tokens x 8 bytes, after the BF16 tile (at most 8 x 128 x 2 bytes).
constexpr uint32_t kTransposeOffset = 4096;
static_assert(kTransposeOffset >= kRows * kBlockN * 2 &&
                  kTransposeOffset + 4 * 32 * kRows * 8 <= kWTileBytes,
              "the transpose buffer lies in W stage 0, past the BF16 tile");
// Folded tiles park pieces' pairs there too: at most F x 128 / F columns x 8
// tokens x 8 bytes = 8 KB.
constexpr uint32_t kParkOffset = kTransposeOffset;
static_assert(kParkOffset + kBlockN * kRows * 8 <= kWTileBytes,
              "the folded pieces' pairs lie in W stage 0, past the BF16 tile");
static_assert(kMaxAccRing % kMaxPipes == 0 && 4 % kMaxPipes == 0,
              "every accumulator slot belongs to one pipe");
static_assert(threads_for_pipes(kMaxPipes) == kMaxThreads && threads_for_pipes(1) == 192,
              "warps 0-5 always, one more MMA-issuing warp per pipe past the first");

// Instruction descriptor of kind::mxf8f6f4 with block scaling: A and B E4M3
// (format 0), both K-major, N = 8 * F (bits 17-22: N >> 3), E8M0 scales
// (bit 23), M = 128 (bits 24-28: M >> 4).  The scale-factor byte ids of A
// (bits 29-30) and B (bits 4-5) select the K block inside a 32-bit scale
// column.
template <int F>
__device__ __forceinline__ uint32_t idesc_for_block(uint32_t kb) {
  constexpr uint32_t kBase = (static_cast<uint32_t>((kRows * F) >> 3) << 17) | (1u << 23) |
                             (static_cast<uint32_t>(kBlockN >> 4) << 24);
  return kBase | (kb << 4) | (kb << 29);
}

// Each BF16 half equal to 0x8000 becomes 0x0000, so no word is the sentinel.
__device__ __forceinline__ uint32_t clear_negative_zero(uint32_t w) {
  uint32_t lo = w & 0xFFFFu, hi = w >> 16;
  lo = (lo == 0x8000u) ? 0u : lo;
  hi = (hi == 0x8000u) ? 0u : hi;
  return lo | (hi << 16);
}

__device__ __forceinline__ void raise_flag(int32_t* state, uint32_t bit) {
  atomicOr(reinterpret_cast<unsigned int*>(state + 3), bit);
}

__device__ __forceinline__ void epilogue_barrier() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

// Compensated summation: (hi, lo) += v with the rounding error of the add
// kept in lo (TwoSum: exact error of a floating-point addition, valid for
// operands of either magnitude order).
__device__ __forceinline__ void two_sum_add(float& hi, float& lo, float v) {
  const float s = __fadd_rn(hi, v);
  const float bp = __fsub_rn(s, hi);
  const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(v, bp));
  hi = s;
  lo = __fadd_rn(lo, err);
}

// BF16 bits of the exact value hi + lo, rounded once to nearest with ties to
// even.  TwoSum gives s = fl(hi + lo) and the exact remainder e with
// |e| <= ulp(s) / 2.  A BF16 midpoint has low 16 bits 0x8000 in FP32, and
// every other FP32 value lies at least one FP32 ulp from the nearest midpoint,
// so s + e rounds as s does unless s is itself a midpoint; there the sign of
// e decides (towards it: away from the midpoint in that direction), and e = 0
// is a true tie.  BF16 being the upper half of FP32, this covers subnormals
// and overflow to infinity alike.
__device__ __forceinline__ uint16_t bf16_bits_from_pair(float hi, float lo) {
  const float s = __fadd_rn(hi, lo);
  const float bp = __fsub_rn(s, hi);
  const float e = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(lo, bp));
  const uint32_t b = __float_as_uint(s);
  if ((b & 0x7F800000u) == 0x7F800000u)  // infinity, or NaN (kept quiet)
    return static_cast<uint16_t>((b >> 16) | ((b & 0x007FFFFFu) != 0u ? 0x0040u : 0u));
  const uint32_t low = b & 0xFFFFu;
  const uint32_t keep = b >> 16;  // sign, exponent and the 7 kept mantissa bits
  bool up;
  if (low != 0x8000u)
    up = low > 0x8000u;
  else if (e == 0.0f)
    up = (keep & 1u) != 0u;
  else
    up = (__float_as_uint(e) >> 31) == (b >> 31);  // e points away from zero
  return static_cast<uint16_t>(keep + (up ? 1u : 0u));  // magnitude + 1 ulp
}

// Position in a ring of mbarrier-guarded slots: the slot and the parity of
// its current use, advanced without divisions in the hot loops.
struct RingCursor {
  int slot;
  uint32_t phase;
  __device__ __forceinline__ void next(int size) {
    if (++slot == size) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// kWideLoad: accumulators read with tcgen05.ld 16x256b (else 32x32b); a
// template parameter so each read-out compiles to its own kernel.  F: the
// fold (K pieces stacked in the MMA's rows).  T: K tiles (of 128 F K each)
// per pipeline stage, 1 or 2 (cta_k 128 or 256): a stage's tiles share one
// full and one empty barrier and come in one W copy, one W-scale copy and
// one x load; accumulator slots, scale slots and the epilogue stay per tile.
template <int S, bool kWideLoad, int F, int T>
__global__ void __launch_bounds__(kMaxThreads, 1)
    publish_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w,
                        const __grid_constant__ CUtensorMap tmap_x,
                        const __grid_constant__ GemmParams p) {
  static_assert(F == 1 || F == 2 || F == 4 || F == 8, "the fold divides the 128 MMA rows");
  static_assert(F == 1 || !kWideLoad, "folded tiles read accumulators with 32x32b");
  static_assert(T == 1 || (T == 2 && !kWideLoad && F <= 4),
                "two K tiles per stage: folds 1, 2, 4 with the 32x32b read-out");
  constexpr int kTileRows = kBlockN / F;                 // output columns of a CTA
  constexpr uint32_t kXStageBytes = kXTileBytes * F;     // F x tiles of 8 x 128 bytes
  constexpr uint32_t kStageTxBytes = kWTileBytes + kXStageBytes + kSfChunkBytes;  // one K tile
  constexpr uint32_t kStageWBytes = kWTileBytes * T;     // a stage's slot in the W ring
  constexpr uint32_t kStageXBytes = kXStageBytes * T;    // ... in the x ring
  constexpr uint32_t kStageSfBytes = kSfChunkBytes * T;  // ... in the W-scale ring
  // x scale chunk of one stage: a 16-byte row per MMA column, 32 rows at most
  // (columns n and n + 32 share row n at fold 8).
  constexpr int kScaleRows = kRows * F < 32 ? kRows * F : 32;
  constexpr int kColsPerScaleRow = (kRows * F + 31) / 32;
  constexpr uint32_t kSxChunkBytes = 16u * kScaleRows;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_addr(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = ptx::smem_addr(smem);
  const GemmSmemLayout& L = p.smem;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t split = (S > 1) ? ptx::cluster_ctarank() : 0u;
  const int tile = blockIdx.x / S;
  const int kt_begin = static_cast<int>(split) * p.tiles_per_split;
  const int kt_end = min(p.k_tiles, kt_begin + p.tiles_per_split);
  const int nkt = max(0, kt_end - kt_begin);  // K tiles of this split
  const int nst = (nkt + T - 1) / T;          // its pipeline stages
  const int stages = p.stages;
  // One accumulator slot per MMA only unfolded (tensor memory holds no ring
  // of 4 x 8F-column slots for F > 1; the host refuses it).
  const bool per_block = F == 1 && p.acc_blocks == 1;
  // `pipes` producer lanes and MMA issuers share the ring, and pipes divides
  // the ring size: then stage i, its slot i % stages, its scale slots and its
  // accumulator slot (the accumulator ring is a multiple of 4) all belong to
  // lane / issuer i % pipes, so every mbarrier is waited on by one thread in
  // use order.  Were a slot to pass between issuers, one could wait on use
  // u + 1 of it before use u completed, while the phase parity it tests still
  // shows the phase before (the parity aliases) and the wait returns at once.
  const int pipes = p.pipes;

  const uint32_t bar_full = sbase + L.bars;                     // [stages]
  const uint32_t bar_empty = bar_full + 8u * stages;            // [stages]
  const int acc_ring = static_cast<int>(p.tmem.acc_ring);
  const uint32_t bar_acc_full = bar_empty + 8u * stages;          // [acc_ring]
  const uint32_t bar_acc_empty = bar_acc_full + 8u * kMaxAccRing;  // [acc_ring]
  const uint32_t bar_sfb = bar_acc_empty + 8u * kMaxAccRing;
  const uint32_t bar_recv = bar_sfb + 8u;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L.misc);  // [0] tmem base, [1] generation

  if (tid == 0) {
    ptx::prefetch_tensormap(&tmap_w);
    ptx::prefetch_tensormap(&tmap_x);
    for (int s = 0; s < stages; ++s) {
      ptx::mbar_init(bar_full + 8u * s, 1);
      ptx::mbar_init(bar_empty + 8u * s, 1);
    }
    for (int r = 0; r < acc_ring; ++r) {
      ptx::mbar_init(bar_acc_full + 8u * r, 1);
      ptx::mbar_init(bar_acc_empty + 8u * r, 128);
    }
    ptx::mbar_init(bar_sfb, 128);
    ptx::mbar_init(bar_recv, 1);
    ptx::fence_mbarrier_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 1) {
    ptx::tmem_alloc(sbase + L.misc, p.tmem.cols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  if (S > 1) {
    ptx::cluster_sync();  // peers' barriers exist before any remote store
  } else {
    __syncthreads();
  }
  ptx::tc_fence_after();
  const uint32_t tmem = misc[0];

  if (warp == 0) {
    // -------------------------------------------------------------- producer
    // The bulk copies one thread issues are served one after another (about
    // 43 GB/s from HBM per issuing thread, whatever the ring depth), so lane
    // l < pipes issues the W tile, W scale chunk and x tile of stages l,
    // l + pipes, l + 2 * pipes, ...
    const int producers = pipes;
    if (lane == 0) ptx::launch_dependents();
    if (lane < producers) {
      if constexpr (T == 1) {
        const uint64_t pol_stream = ptx::policy_evict_first();
        const uint64_t pol_keep = ptx::policy_evict_last();
        const int npre = min(stages, nkt);
        // One 16 KB W stage (F pieces of R rows x 128 bytes, 128 rows in all):
        // a contiguous image from the tiled copy, or F 2-D TMA boxes (with the
        // same 128-byte swizzle) of W in place.
        auto load_w_tile = [&](uint32_t dst, int kt, uint32_t bar) {
          if (p.w_tiled != nullptr) {
            ptx::bulk_load(dst, p.w_tiled + (static_cast<size_t>(tile) * p.k_tiles + kt) * kWTileBytes,
                           kWTileBytes, bar, pol_stream);
          } else {
  #pragma unroll
            for (int pc = 0; pc < F; ++pc)
              ptx::tma_load_2d(dst + pc * (kTileRows * kTileK), &tmap_w, (kt * F + pc) * kTileK,
                               tile * kTileRows, bar, pol_stream);
          }
        };
        // The F activation tiles of a stage, rows >= m read as zero: one box of
        // the 3-D piece view (128 K x 8 rows x F pieces, piece-major in shared
        // memory, as F boxes of the 2-D view would land), or F 2-D boxes.
        auto load_x_tile = [&](uint32_t dst, int kt, uint32_t bar) {
          if (F > 1 && p.x_pieces) {
            ptx::tma_load_3d(dst, &tmap_x, 0, 0, kt * F, bar, pol_keep);
          } else {
  #pragma unroll
            for (int pc = 0; pc < F; ++pc)
              ptx::tma_load_2d(dst + pc * kXTileBytes, &tmap_x, (kt * F + pc) * kTileK, 0, bar,
                               pol_keep);
          }
        };
        // W and its scales do not depend on the previous kernel: start them now.
        for (int i = lane; i < npre; i += producers) {
          const uint32_t full = bar_full + 8u * i;
          const int kt = kt_begin + i;
          ptx::mbar_arrive_expect_tx(full, kStageTxBytes);
          load_w_tile(sbase + L.w + i * kWTileBytes, kt, full);
          ptx::bulk_load(sbase + L.sfa + i * kSfChunkBytes,
                         p.w_sf + (static_cast<size_t>(tile) * p.k_tiles + kt) * kSfChunkBytes,
                         kSfChunkBytes, full, pol_stream);
        }
        // Warm L2 with the stages that come after the ring, so HBM keeps
        // streaming while the previous kernel finishes and the grid wait holds.
        // The first CTAs of the grid launch while the previous kernel still
        // streams (its dependents launch as soon as it starts), so they warm
        // fewer stages and leave it the bandwidth; the later ones, which start
        // as its CTAs exit, warm more and bridge the hand-over.
        const int depth = static_cast<int>(blockIdx.x) < p.early_ctas ? p.l2_prefetch_early
                                                                       : p.l2_prefetch;
        const int nwarm = min(nkt, npre + depth);
        if (lane == 0 && nwarm > npre) {
          if (p.w_tiled != nullptr) {
            ptx::prefetch_l2(p.w_tiled + (static_cast<size_t>(tile) * p.k_tiles + kt_begin + npre) *
                                             kWTileBytes,
                             static_cast<uint32_t>(nwarm - npre) * kWTileBytes);
          } else {
            for (int i = npre; i < nwarm; ++i)
  #pragma unroll
              for (int pc = 0; pc < F; ++pc)
                ptx::prefetch_l2_tile(&tmap_w, ((kt_begin + i) * F + pc) * kTileK,
                                      tile * kTileRows);
          }
          ptx::prefetch_l2(p.w_sf + (static_cast<size_t>(tile) * p.k_tiles + kt_begin + npre) *
                                        kSfChunkBytes,
                           static_cast<uint32_t>(nwarm - npre) * kSfChunkBytes);
        }
        // The activations follow the programmatic grid wait.
        ptx::grid_dependency_wait();
        for (int i = lane; i < npre; i += producers)
          load_x_tile(sbase + L.x + i * kXStageBytes, kt_begin + i, bar_full + 8u * i);
        // From here every slot is on its second or later use: wait until the
        // MMAs of its previous use released it.  This lane's stages advance the
        // ring by `producers` slots at a time.
        int issued = -1;  // the last stage this lane issued
        for (int i = lane; i < npre; i += producers) issued = i;
        const int first = npre + ((lane - npre % producers) % producers + producers) % producers;
        RingCursor ring{first - npre, 1u};  // npre == stages whenever this loop runs
        for (int i = first; i < nkt; i += producers) {
          const int s = ring.slot;
          if (!ptx::mbar_wait(bar_empty + 8u * s, ring.phase ^ 1u, p.wait_limit_ns)) {
            raise_flag(p.state, 0x2u);
            break;
          }
          const uint32_t full = bar_full + 8u * s;
          const int kt = kt_begin + i;
          ptx::mbar_arrive_expect_tx(full, kStageTxBytes);
          load_w_tile(sbase + L.w + s * kWTileBytes, kt, full);
          ptx::bulk_load(sbase + L.sfa + s * kSfChunkBytes,
                         p.w_sf + (static_cast<size_t>(tile) * p.k_tiles + kt) * kSfChunkBytes,
                         kSfChunkBytes, full, pol_stream);
          load_x_tile(sbase + L.x + s * kXStageBytes, kt, full);
          issued = i;
          ring.slot += producers;
          if (ring.slot >= stages) {
            ring.slot -= stages;
            ring.phase ^= 1u;
          }
        }
        // This lane's copies still in flight land before the CTA leaves
        // (immediate when the MMAs consumed them, which is the normal case):
        // its stages among the last `stages` of the split, the latest use of
        // their slots (no stage past nkt - 1 reuses them, so each wait is on
        // the phase of this lane's own copy).
        for (int i = issued; i >= max(0, nkt - stages); i -= producers)
          ptx::mbar_wait(bar_full + 8u * (i % stages), static_cast<uint32_t>(i / stages) & 1u,
                         p.wait_limit_ns);
      } else {
        const uint64_t pol_stream = ptx::policy_evict_first();
        const uint64_t pol_keep = ptx::policy_evict_last();
        const int npre = min(stages, nst);
        // A stage's W: nt 16 KB tiles (F pieces of R rows x 128 bytes, 128 rows
        // each), a contiguous image from the tiled copy, or F 2-D TMA boxes per
        // tile (with the same 128-byte swizzle) of W in place; and their scale
        // chunks, contiguous in the re-laid copy.
        auto load_w_stage = [&](uint32_t slot, int kt0, int nt, uint32_t bar) {
          if (p.w_tiled != nullptr) {
            ptx::bulk_load(sbase + L.w + slot * kStageWBytes,
                           p.w_tiled + (static_cast<size_t>(tile) * p.k_tiles + kt0) * kWTileBytes,
                           static_cast<uint32_t>(nt) * kWTileBytes, bar, pol_stream);
          } else {
            for (int t = 0; t < nt; ++t)
  #pragma unroll
              for (int pc = 0; pc < F; ++pc)
                ptx::tma_load_2d(sbase + L.w + slot * kStageWBytes + t * kWTileBytes +
                                     pc * (kTileRows * kTileK),
                                 &tmap_w, ((kt0 + t) * F + pc) * kTileK, tile * kTileRows, bar,
                                 pol_stream);
          }
          ptx::bulk_load(sbase + L.sfa + slot * kStageSfBytes,
                         p.w_sf + (static_cast<size_t>(tile) * p.k_tiles + kt0) * kSfChunkBytes,
                         static_cast<uint32_t>(nt) * kSfChunkBytes, bar, pol_stream);
        };
        // A stage's x: its T tiles of F pieces each (T x F 8 x 128-byte boxes,
        // rows >= m and pieces past K read as zero): one box of the 3-D piece
        // view (128 K x 8 rows x T F pieces, piece-major in shared memory, as
        // the 2-D boxes would land), or T F boxes of the 2-D view.  A stage
        // with fewer than T tiles left still loads T tiles of x (zeros, or the
        // next split's, unused), so its byte count is fixed.
        auto load_x_stage = [&](uint32_t slot, int kt0, uint32_t bar) {
          const uint32_t dst = sbase + L.x + slot * kStageXBytes;
          if (F * T > 1 && p.x_pieces) {
            ptx::tma_load_3d(dst, &tmap_x, 0, 0, kt0 * F, bar, pol_keep);
          } else {
  #pragma unroll
            for (int pc = 0; pc < F * T; ++pc)
              ptx::tma_load_2d(dst + pc * kXTileBytes, &tmap_x, (kt0 * F + pc) * kTileK, 0, bar,
                               pol_keep);
          }
        };
        auto stage_tiles = [&](int i) { return min(T, nkt - i * T); };
        auto stage_bytes = [&](int nt) {
          return static_cast<uint32_t>(nt) * (kWTileBytes + kSfChunkBytes) + kStageXBytes;
        };
        // W and its scales do not depend on the previous kernel: start them now.
        for (int i = lane; i < npre; i += producers) {
          const uint32_t full = bar_full + 8u * i;
          ptx::mbar_arrive_expect_tx(full, stage_bytes(stage_tiles(i)));
          load_w_stage(i, kt_begin + i * T, stage_tiles(i), full);
        }
        // Warm L2 with the stages that come after the ring, so HBM keeps
        // streaming while the previous kernel finishes and the grid wait holds.
        // The first CTAs of the grid launch while the previous kernel still
        // streams (its dependents launch as soon as it starts), so they warm
        // fewer stages and leave it the bandwidth; the later ones, which start
        // as its CTAs exit, warm more and bridge the hand-over.
        const int depth = static_cast<int>(blockIdx.x) < p.early_ctas ? p.l2_prefetch_early
                                                                       : p.l2_prefetch;
        const int warm_begin = npre * T;                       // K tiles of the split
        const int warm_end = min(nkt, (npre + depth) * T);
        if (lane == 0 && warm_end > warm_begin) {
          if (p.w_tiled != nullptr) {
            ptx::prefetch_l2(p.w_tiled + (static_cast<size_t>(tile) * p.k_tiles + kt_begin +
                                          warm_begin) * kWTileBytes,
                             static_cast<uint32_t>(warm_end - warm_begin) * kWTileBytes);
          } else {
            for (int i = warm_begin; i < warm_end; ++i)
  #pragma unroll
              for (int pc = 0; pc < F; ++pc)
                ptx::prefetch_l2_tile(&tmap_w, ((kt_begin + i) * F + pc) * kTileK,
                                      tile * kTileRows);
          }
          ptx::prefetch_l2(p.w_sf + (static_cast<size_t>(tile) * p.k_tiles + kt_begin +
                                     warm_begin) * kSfChunkBytes,
                           static_cast<uint32_t>(warm_end - warm_begin) * kSfChunkBytes);
        }
        // The activations follow the programmatic grid wait.
        ptx::grid_dependency_wait();
        for (int i = lane; i < npre; i += producers)
          load_x_stage(i, kt_begin + i * T, bar_full + 8u * i);
        // From here every slot is on its second or later use: wait until the
        // MMAs of its previous use released it.  This lane's stages advance the
        // ring by `producers` slots at a time.
        int issued = -1;  // the last stage this lane issued
        for (int i = lane; i < npre; i += producers) issued = i;
        const int first = npre + ((lane - npre % producers) % producers + producers) % producers;
        RingCursor ring{first - npre, 1u};  // npre == stages whenever this loop runs
        for (int i = first; i < nst; i += producers) {
          const int s = ring.slot;
          if (!ptx::mbar_wait(bar_empty + 8u * s, ring.phase ^ 1u, p.wait_limit_ns)) {
            raise_flag(p.state, 0x2u);
            break;
          }
          const uint32_t full = bar_full + 8u * s;
          const int kt0 = kt_begin + i * T;
          ptx::mbar_arrive_expect_tx(full, stage_bytes(stage_tiles(i)));
          load_w_stage(s, kt0, stage_tiles(i), full);
          load_x_stage(s, kt0, full);
          issued = i;
          ring.slot += producers;
          if (ring.slot >= stages) {
            ring.slot -= stages;
            ring.phase ^= 1u;
          }
        }
        // This lane's copies still in flight land before the CTA leaves
        // (immediate when the MMAs consumed them, which is the normal case):
        // its stages among the last `stages` of the split, the latest use of
        // their slots (no stage past nkt - 1 reuses them, so each wait is on
        // the phase of this lane's own copy).
        for (int i = issued; i >= max(0, nst - stages); i -= producers)
          ptx::mbar_wait(bar_full + 8u * (i % stages), static_cast<uint32_t>(i / stages) & 1u,
                         p.wait_limit_ns);
      }
    }
  } else if (warp == 1 || warp >= 6) {
    const int issuer = warp == 1 ? 0 : warp - 5;
    if (lane == 0 && issuer < pipes) {
      // --------------------------------------------------------- MMA issuers
      // tcgen05 instructions cost their issuing thread a fixed time each
      // (about 260 ns per 16 KB stage of 2 copies, 4 MMAs and 2 commits),
      // which caps one thread near 65 GB/s of weight, so issuer j < pipes
      // takes stages j, j + pipes, ...
      ptx::grid_dependency_wait();
      bool ok = true;
      if (nkt > 0) {
        ok = ptx::mbar_wait(bar_sfb, 0, p.wait_limit_ns);
        if (!ok) raise_flag(p.state, 0x2u);
        ptx::tc_fence_after();
      }
      if constexpr (T == 1) {
        RingCursor stage{0, 0u}, acc{0, 0u};
        for (int q = 0; q < issuer; ++q) {
          stage.next(stages);
          acc.next(acc_ring);
        }
        for (int i = issuer; i < nkt && ok; i += pipes) {
          const int s = stage.slot;
          const int r = acc.slot;
          if (!ptx::mbar_wait(bar_full + 8u * s, stage.phase, p.wait_limit_ns) ||
              (i >= acc_ring &&
               !ptx::mbar_wait(bar_acc_empty + 8u * r, acc.phase ^ 1u, p.wait_limit_ns))) {
            raise_flag(p.state, 0x2u);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sfa_t = tmem + p.tmem.sfa + 4u * s;
          const uint32_t sfb_t = tmem + p.tmem.sfb + 4u * s;
          ptx::tmem_cp_32x128b_warpx4(sfa_t, ptx::desc_rows16(sbase + L.sfa + s * kSfChunkBytes));
          ptx::tmem_cp_32x128b_warpx4(sfb_t, ptx::desc_rows16(sbase + L.sx + i * kSxChunkBytes));
          const uint32_t a0 = sbase + L.w + s * kWTileBytes;
          const uint32_t b0 = sbase + L.x + s * kXStageBytes;
          const uint32_t d0 = tmem + p.tmem.acc + p.tmem.acc_slot * static_cast<uint32_t>(r);
  #pragma unroll
          for (uint32_t kb = 0; kb < kSfPerTile; ++kb) {
            // One 8-column accumulator per block, or one per stage.
            const uint32_t d = per_block ? d0 + 8u * kb : d0;
            const uint32_t accumulate = per_block ? 0u : (kb > 0 ? 1u : 0u);
            ptx::mma_mxf8(d, ptx::desc_kmajor_sw128(a0 + 32u * kb),
                          ptx::desc_kmajor_sw128(b0 + 32u * kb), idesc_for_block<F>(kb),
                          accumulate, sfa_t, sfb_t);
          }
          ptx::mma_commit(bar_empty + 8u * s);
          ptx::mma_commit(bar_acc_full + 8u * r);
          for (int q = 0; q < pipes; ++q) {
            stage.next(stages);
            acc.next(acc_ring);
          }
        }
      } else {
        // Issuer j takes stages j, j + pipes, ...; a stage's tiles take
        // consecutive accumulator slots and scale slots (the accumulator ring is
        // a multiple of T pipes, so every slot keeps one issuer).
        RingCursor stage{0, 0u}, acc{0, 0u};
        for (int q = 0; q < issuer; ++q) stage.next(stages);
        for (int q = 0; q < issuer * T; ++q) acc.next(acc_ring);
        for (int i = issuer; i < nst && ok; i += pipes) {
          const int s = stage.slot;
          if (!ptx::mbar_wait(bar_full + 8u * s, stage.phase, p.wait_limit_ns)) {
            raise_flag(p.state, 0x2u);
            ok = false;
            break;
          }
          const int nt = min(T, nkt - i * T);
  #pragma unroll
          for (int t = 0; t < T; ++t) {
            if (t >= nt) break;
            const int j = i * T + t;  // K tile of the split
            const int r = acc.slot;
            if (j >= acc_ring &&
                !ptx::mbar_wait(bar_acc_empty + 8u * r, acc.phase ^ 1u, p.wait_limit_ns)) {
              raise_flag(p.state, 0x2u);
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t sc = static_cast<uint32_t>(s * T + t);  // scale slot of the tile
            const uint32_t sfa_t = tmem + p.tmem.sfa + 4u * sc;
            const uint32_t sfb_t = tmem + p.tmem.sfb + 4u * sc;
            ptx::tmem_cp_32x128b_warpx4(sfa_t, ptx::desc_rows16(sbase + L.sfa + sc * kSfChunkBytes));
            ptx::tmem_cp_32x128b_warpx4(sfb_t, ptx::desc_rows16(sbase + L.sx + j * kSxChunkBytes));
            const uint32_t a0 = sbase + L.w + s * kStageWBytes + t * kWTileBytes;
            const uint32_t b0 = sbase + L.x + s * kStageXBytes + t * kXStageBytes;
            const uint32_t d0 = tmem + p.tmem.acc + p.tmem.acc_slot * static_cast<uint32_t>(r);
  #pragma unroll
            for (uint32_t kb = 0; kb < kSfPerTile; ++kb) {
              // One 8-column accumulator per block, or one per tile.
              const uint32_t d = per_block ? d0 + 8u * kb : d0;
              const uint32_t accumulate = per_block ? 0u : (kb > 0 ? 1u : 0u);
              ptx::mma_mxf8(d, ptx::desc_kmajor_sw128(a0 + 32u * kb),
                            ptx::desc_kmajor_sw128(b0 + 32u * kb), idesc_for_block<F>(kb),
                            accumulate, sfa_t, sfb_t);
            }
            if (t + 1 == nt) ptx::mma_commit(bar_empty + 8u * s);  // the stage's last tile
            ptx::mma_commit(bar_acc_full + 8u * r);
            acc.next(acc_ring);
          }
          for (int q = 0; q < pipes; ++q) stage.next(stages);
          for (int q = nt; q < pipes * T; ++q) acc.next(acc_ring);  // the other issuers' tiles
        }
      }
    }
  }
  if (warp < 2 || warp >= 6) {
    __syncwarp();
    if (S > 1) {
      if (!p.smem.recv_dedicated)
        ptx::cluster_sync();  // matches the epilogue's barrier before the exchange
      ptx::cluster_arrive();  // these warps address no peer: the final barrier's arrival
    }
  } else {
    // ------------------------------------------------------------- epilogue
    const int etid = tid - 64;               // 0..127
    const int quarter = warp & 3;            // the 32 TMEM lanes this warp reaches
    const int arow = quarter * 32 + lane;    // MMA row = TMEM lane
    const int piece = F == 1 ? 0 : arow / kTileRows;     // the K piece this lane holds
    const int col = F == 1 ? arow : arow % kTileRows;    // output column within the tile
    // The lane's diagonal block is columns [8 piece, 8 piece + 8) of a slot.
    // A tensor-memory load takes one address for the whole warp: up to F = 4 a
    // warp's 32 lanes hold one piece; at F = 8 they hold two (16 rows each),
    // so the warp loads both blocks (16 columns) and each lane keeps its own.
    constexpr int kPiecesPerWarp = F == 8 ? 2 : 1;
    const int warp_piece = F == 1 ? 0 : (quarter * 32) / kTileRows;  // the warp's first piece
    const uint32_t lane_base =
        (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(kRows * warp_piece);
    ptx::grid_dependency_wait();
    if (etid == 0) misc[1] = ptx::ld_volatile_u32(p.state + 0);

    // x scales of this CTA's K range as one chunk per stage: MMA column r
    // (token r % 8 of piece r / 8) at row r % 32 of stage j's chunk (byte
    // j * kSxChunkBytes + (r % 32) * 16), its four E8M0 codes at bytes
    // 4 (r / 32) .. +3 of the row (the 32x128b copy's layout: at fold 8 a
    // row holds columns r and r + 32), the rest of the row zero.  Tokens >= m
    // and blocks past K take 127 (a scale of 1; those x elements are zero).
    // The copy of a chunk reads 32 rows; rows past the chunk (the next
    // chunks, or the tail) feed no kept column.  (Loading every word into
    // registers before any store measured 2-6 % slower per call than this
    // loop.)
    uint8_t* sx = smem + L.sx;
    const int kblocks = p.k / 32;
    const int words = kScaleRows * nkt;  // <= 8 x kMaxTilesPerSplit (host check)
    constexpr int kMaxWords = kRows * kMaxTilesPerSplit / 128;  // per thread
#pragma unroll
    for (int it = 0; it < kMaxWords; ++it) {
      const int w = etid + it * 128;
      if (w >= words) break;
      const int n0 = w / nkt;
      const int j = w - n0 * nkt;
      uint32_t v[2] = {0u, 0u};
#pragma unroll
      for (int n1 = 0; n1 < kColsPerScaleRow; ++n1) {
        const int r = n0 + 32 * n1;
        const int t = F == 1 ? r : r % kRows;
        v[n1] = 0x7F7F7F7Fu;
        if (t < p.m) {
          const int kb0 = ((kt_begin + j) * F + (F == 1 ? 0 : r / kRows)) * kSfPerTile;
          const uint8_t* row = p.x_scale + static_cast<size_t>(t) * kblocks;
          uint32_t b[kSfPerTile];
#pragma unroll
          for (int q = 0; q < kSfPerTile; ++q) b[q] = kb0 + q < kblocks ? row[kb0 + q] : 127u;
          v[n1] = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
        }
      }
      *reinterpret_cast<uint4*>(sx + j * kSxChunkBytes + n0 * 16) =
          make_uint4(v[0], v[1], 0u, 0u);
    }
    ptx::fence_proxy_async_smem();  // the tensor-memory copy reads them
    ptx::mbar_arrive(bar_sfb);

    // Fold every completed accumulator slot into the compensated sums.  With
    // the 32x32b load thread = output column and hi[t] / lo[t] hold token t;
    // with the 16x256b load (two per slot, lane halves 0-15 and 16-31 of the
    // warp's quarter) element a = 4 h + r of a thread holds column
    // 16 h + 8 (r / 2) + lane / 4 of the quarter and token 2 (lane % 4) +
    // r % 2, and one warp-local transpose after the loop brings back the
    // column-per-thread layout.  Each element sees the same values in the same
    // order either way, so the two loads give identical bits.
    constexpr bool wide_load = kWideLoad;
    float hi[kRows], lo[kRows];
#pragma unroll
    for (int t = 0; t < kRows; ++t) hi[t] = lo[t] = 0.0f;
    RingCursor acc{0, 0u};
    for (int i = 0; i < nkt; ++i, acc.next(acc_ring)) {
      const int r = acc.slot;
      if (!ptx::mbar_wait(bar_acc_full + 8u * r, acc.phase, p.wait_limit_ns)) {
        raise_flag(p.state, 0x2u);
        break;
      }
      ptx::tc_fence_after();
      const uint32_t slot =
          tmem + lane_base + p.tmem.acc + p.tmem.acc_slot * static_cast<uint32_t>(r);
      if constexpr (wide_load) {
        constexpr uint32_t kHalf = 16u << 16;  // lane offset of the second half
        if (per_block) {
          uint32_t v0[16], v1[16];
          ptx::tmem_ld_16x256b_x4(slot, v0);
          ptx::tmem_ld_16x256b_x4(slot + kHalf, v1);
          ptx::tmem_wait_ld();
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar_acc_empty + 8u * r);
#pragma unroll
          for (int kb = 0; kb < kSfPerTile; ++kb)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              two_sum_add(hi[e], lo[e], __uint_as_float(v0[kb * 4 + e]));
              two_sum_add(hi[4 + e], lo[4 + e], __uint_as_float(v1[kb * 4 + e]));
            }
        } else {
          uint32_t v0[4], v1[4];
          ptx::tmem_ld_16x256b_x1(slot, v0);
          ptx::tmem_ld_16x256b_x1(slot + kHalf, v1);
          ptx::tmem_wait_ld();
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar_acc_empty + 8u * r);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            two_sum_add(hi[e], lo[e], __uint_as_float(v0[e]));
            two_sum_add(hi[4 + e], lo[4 + e], __uint_as_float(v1[e]));
          }
        }
      } else if (per_block) {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(slot, v);
        ptx::tmem_wait_ld();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar_acc_empty + 8u * r);
#pragma unroll
        for (int kb = 0; kb < kSfPerTile; ++kb)
#pragma unroll
          for (int t = 0; t < kRows; ++t)
            two_sum_add(hi[t], lo[t], __uint_as_float(v[kb * 8 + t]));
      } else if constexpr (kPiecesPerWarp == 2) {
        uint32_t v[16];
        ptx::tmem_ld_32x32b_x16(slot, v);
        ptx::tmem_wait_ld();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar_acc_empty + 8u * r);
        const bool second = piece != warp_piece;
#pragma unroll
        for (int t = 0; t < kRows; ++t)
          two_sum_add(hi[t], lo[t], __uint_as_float(second ? v[kRows + t] : v[t]));
      } else {
        uint32_t v[8];
        ptx::tmem_ld_32x32b_x8(slot, v);
        ptx::tmem_wait_ld();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar_acc_empty + 8u * r);
#pragma unroll
        for (int t = 0; t < kRows; ++t) two_sum_add(hi[t], lo[t], __uint_as_float(v[t]));
      }
    }

    if constexpr (wide_load) {
      // Transpose through this warp's 2 KB of the dead W stage 0 (past the
      // BF16 tile): [column of the quarter][token] pairs.
      float2* pairs = reinterpret_cast<float2*>(smem + L.w + kTransposeOffset) + quarter * 32 * kRows;
#pragma unroll
      for (int a = 0; a < kRows; ++a) {
        const int c = (a / 4) * 16 + ((a % 4) / 2) * 8 + lane / 4;
        const int t = 2 * (lane % 4) + (a % 2);
        pairs[c * kRows + t] = make_float2(hi[a], lo[a]);
      }
      __syncwarp();
#pragma unroll
      for (int t = 0; t < kRows; ++t) {
        const float2 v = pairs[lane * kRows + t];
        hi[t] = v.x;
        lo[t] = v.y;
      }
    }

    // Folded tiles: the F lanes that hold one output column (one K piece
    // each) add its pieces in piece order, the pairs passing through W stage
    // 0 (dead: every MMA of this CTA has completed), past the BF16 tile: lane
    // p of a column takes its tokens [p 8/F, (p+1) 8/F), parks the pairs of the
    // others ([piece][column][token]) and adds the F pieces of its own.  With
    // split-K it then sends each of its tokens that another CTA owns to the
    // same lane of that CTA, and finishes those its own CTA owns.  The
    // additions run in piece order, then K-slice order, whichever lane does
    // them.
    constexpr int kShard = kRows / S;  // tokens this CTA finishes
    static_assert(kShard * S == kRows && (kShard == 1 || kShard % 2 == 0),
                  "tokens split evenly, in pairs or one per CTA");
    uint16_t* ctile = reinterpret_cast<uint16_t*>(smem + L.ctile);  // [kShard][kTileRows]
    if constexpr (F > 1) {
      constexpr int kPerLane = kRows / F;  // tokens a lane adds the pieces of
      float2* park = reinterpret_cast<float2*>(smem + L.w + kParkOffset);
#pragma unroll
      for (int t = 0; t < kRows; ++t)
        if (t / kPerLane != piece)
          park[(piece * kTileRows + col) * kRows + t] = make_float2(hi[t], lo[t]);
      epilogue_barrier();
      float red_hi[kPerLane], red_lo[kPerLane];  // tokens piece * kPerLane + j
#pragma unroll
      for (int j = 0; j < kPerLane; ++j) {
        float oh = 0.0f, ol = 0.0f;  // this lane's own pair of the token
#pragma unroll
        for (int t = j; t < kRows; t += kPerLane)
          if (t / kPerLane == piece) {
            oh = hi[t];
            ol = lo[t];
          }
        const int t = piece * kPerLane + j;
        float sh = 0.0f, sl = 0.0f;
#pragma unroll
        for (int q = 0; q < F; ++q) {
          float vh = oh, vl = ol;
          if (q != piece) {
            const float2 v = park[(q * kTileRows + col) * kRows + t];
            vh = v.x;
            vl = v.y;
          }
          if (q == 0) {
            sh = vh;
            sl = vl;
          } else {
            two_sum_add(sh, sl, vh);
            sl = __fadd_rn(sl, vl);
          }
        }
        red_hi[j] = sh;
        red_lo[j] = sl;
      }
      const float a = p.alpha != nullptr ? *p.alpha : 1.0f;
      // The global scale and the one rounding of a finished token (as below).
      auto finish = [&](int t_local, float sh, float sl) {
        if (p.alpha != nullptr) {
          const float ph = __fmul_rn(a, sh);
          const float pe = __fmaf_rn(a, sh, -ph);
          sl = __fmaf_rn(a, sl, pe);
          sh = ph;
        }
        ctile[t_local * kTileRows + col] = bf16_bits_from_pair(sh, sl);
      };
      if constexpr (S == 1) {
#pragma unroll
        for (int j = 0; j < kPerLane; ++j) finish(piece * kPerLane + j, red_hi[j], red_lo[j]);
      } else {
        // A lane's tokens fall in runs of kRun that one CTA owns; the receive
        // buffer is [sender][MMA row][kRun pairs], the MMA row naming the lane.
        constexpr int kRun = kPerLane < kShard ? kPerLane : kShard;
        constexpr int kRuns = kPerLane / kRun;
        static_assert(kRun % 2 == 0, "runs go out as 16-byte stores of two pairs");
        // A receive buffer in the W ring is dead only once every CTA of the
        // cluster has finished its main loop; one of its own needs no barrier
        // (a peer's bytes may land before this CTA's expect: the transaction
        // count runs negative until then).
        if (!p.smem.recv_dedicated) ptx::cluster_sync();
        if (etid == 0)
          ptx::mbar_arrive_expect_tx(bar_recv,
                                     static_cast<uint32_t>((S - 1) * kTileRows * kShard * 8));
        const int sender = static_cast<int>(split);
#pragma unroll
        for (int r = 0; r < kRuns; ++r) {
          const int dest = (piece * kPerLane + r * kRun) / kShard;
          if (dest == sender) continue;
          const int sidx = sender < dest ? sender : sender - 1;
          const uint32_t remote_bar = ptx::map_to_rank(bar_recv, dest);
          const uint32_t remote =
              ptx::map_to_rank(sbase + L.recv + (sidx * kBlockN + arow) * kRun * 8, dest);
#pragma unroll
          for (int j = 0; j < kRun; j += 2)
            ptx::st_async_remote_v4(
                remote + j * 8,
                make_uint4(__float_as_uint(red_hi[r * kRun + j]), __float_as_uint(red_lo[r * kRun + j]),
                           __float_as_uint(red_hi[r * kRun + j + 1]),
                           __float_as_uint(red_lo[r * kRun + j + 1])),
                remote_bar);
        }
        // This thread addresses no peer after its sends: its half of the final
        // cluster barrier, whose wait comes before the CTA exits.
        ptx::cluster_arrive();
        if (!ptx::mbar_wait_cluster(bar_recv, 0, p.wait_limit_ns)) raise_flag(p.state, 0x2u);
        const float2* recv = reinterpret_cast<const float2*>(smem + L.recv);
#pragma unroll
        for (int r = 0; r < kRuns; ++r) {
          if ((piece * kPerLane + r * kRun) / kShard != sender) continue;
#pragma unroll
          for (int j = 0; j < kRun; ++j) {
            float sh = 0.0f, sl = 0.0f;
#pragma unroll
            for (int src = 0; src < S; ++src) {
              float vh = red_hi[r * kRun + j], vl = red_lo[r * kRun + j];
              if (src != sender) {
                const int sidx = src < sender ? src : src - 1;
                const float2 v = recv[(sidx * kBlockN + arow) * kRun + j];
                vh = v.x;
                vl = v.y;
              }
              two_sum_add(sh, sl, vh);
              sl = __fadd_rn(sl, vl);
            }
            finish(piece * kPerLane + r * kRun + j - sender * kShard, sh, sl);
          }
        }
      }
    } else {
      // Split-K: every CTA sends the (hi, lo) pairs of the tokens it does not
      // own to their owners, then sums the S pairs of its own tokens in K-slice
      // order.  A split with no K tiles contributes zeros.  The receive buffer
      // is [sender][column][token][hi, lo]: one CTA's pairs for one column are
      // 8 * kShard contiguous bytes, sent as 16-byte stores (8-byte ones at
      // S = 8, where each CTA owns one token).
      float own_hi[kShard], own_lo[kShard];
      if constexpr (S > 1) {
        constexpr int kPairBytes = kShard * 8;
        // A receive buffer in the W ring is dead only once every CTA of the
        // cluster has finished its main loop; one of its own needs no barrier
        // (a peer's bytes may land before this CTA's expect: the transaction
        // count runs negative until then).
        if (!p.smem.recv_dedicated) ptx::cluster_sync();
        if (etid == 0)
          ptx::mbar_arrive_expect_tx(bar_recv,
                                     static_cast<uint32_t>((S - 1) * kTileRows * kPairBytes));
#pragma unroll
        for (int peer = 0; peer < S; ++peer) {
          if (peer == static_cast<int>(split)) continue;
          const int sender = static_cast<int>(split) < peer ? static_cast<int>(split)
                                                            : static_cast<int>(split) - 1;
          const uint32_t remote_bar = ptx::map_to_rank(bar_recv, peer);
          const uint32_t remote =
              ptx::map_to_rank(sbase + L.recv + (sender * kTileRows + col) * kPairBytes, peer);
          if constexpr (kShard == 1) {
            ptx::st_async_remote_v2(remote, __float_as_uint(hi[peer]), __float_as_uint(lo[peer]),
                                    remote_bar);
          } else {
#pragma unroll
            for (int jj = 0; jj < kShard; jj += 2)
              ptx::st_async_remote_v4(
                  remote + jj * 8,
                  make_uint4(__float_as_uint(hi[peer * kShard + jj]),
                             __float_as_uint(lo[peer * kShard + jj]),
                             __float_as_uint(hi[peer * kShard + jj + 1]),
                             __float_as_uint(lo[peer * kShard + jj + 1])),
                  remote_bar);
          }
        }
        // This thread addresses no peer after its sends: its half of the final
        // cluster barrier, whose wait comes before the CTA exits.
        ptx::cluster_arrive();
        if (!ptx::mbar_wait_cluster(bar_recv, 0, p.wait_limit_ns)) raise_flag(p.state, 0x2u);
        const uint8_t* recv = smem + L.recv;
#pragma unroll
        for (int jj = 0; jj < kShard; ++jj) {
          float sh = 0.0f, sl = 0.0f;
#pragma unroll
          for (int src = 0; src < S; ++src) {
            float vh, vl;
            if (src == static_cast<int>(split)) {
              vh = 0.0f;
              vl = 0.0f;
#pragma unroll
              for (int q = 0; q < kRows; ++q)
                if (q == static_cast<int>(split) * kShard + jj) {
                  vh = hi[q];
                  vl = lo[q];
                }
            } else {
              const int sidx = src < static_cast<int>(split) ? src : src - 1;
              const float2 pair = *reinterpret_cast<const float2*>(
                  recv + (sidx * kTileRows + col) * kPairBytes + jj * 8);
              vh = pair.x;
              vl = pair.y;
            }
            two_sum_add(sh, sl, vh);
            sl = __fadd_rn(sl, vl);
          }
          own_hi[jj] = sh;
          own_lo[jj] = sl;
        }
      } else {
#pragma unroll
        for (int jj = 0; jj < kShard; ++jj) {
          own_hi[jj] = hi[jj];
          own_lo[jj] = lo[jj];
        }
      }

      // The global scale (gemm page, epilog_warp with use_scale: the
      // accumulator times mScale[0]) multiplies the compensated sum before its
      // one rounding: alpha * hi exactly as a product and its FMA error, plus
      // alpha * lo.  It is read after the grid wait like x.
      if (p.alpha != nullptr) {
        const float a = *p.alpha;
#pragma unroll
        for (int jj = 0; jj < kShard; ++jj) {
          const float ph = __fmul_rn(a, own_hi[jj]);
          const float pe = __fmaf_rn(a, own_hi[jj], -ph);
          own_lo[jj] = __fmaf_rn(a, own_lo[jj], pe);
          own_hi[jj] = ph;
        }
      }

#pragma unroll
      for (int jj = 0; jj < kShard; ++jj)
        ctile[jj * kTileRows + col] = bf16_bits_from_pair(own_hi[jj], own_lo[jj]);
    }
    epilogue_barrier();

    const uint32_t g = misc[1];
    const bool generation_ok = g < static_cast<uint32_t>(kGenerations);
    const size_t n0 = static_cast<size_t>(tile) * kTileRows;
    for (int pk = etid; pk < kShard * (kTileRows / 8); pk += 128) {
      const int jj = pk / (kTileRows / 8);
      const int chunk = pk % (kTileRows / 8);
      const int t = static_cast<int>(split) * kShard + jj;
      if (t >= p.m) continue;
      const uint4 v = *reinterpret_cast<const uint4*>(ctile + jj * kTileRows + chunk * 8);
      const size_t column = n0 + chunk * 8;
      if (p.c != nullptr) ptx::st_v4(p.c + static_cast<size_t>(t) * p.n + column, v);
      if (p.publish && generation_ok) {
        const uint4 clean = make_uint4(clear_negative_zero(v.x), clear_negative_zero(v.y),
                                       clear_negative_zero(v.z), clear_negative_zero(v.w));
        ptx::st_v4(p.mailbox + (static_cast<size_t>(g) * p.capacity + t) * p.n + column, clean);
      }
    }
    // Hand the generation to the consumer, once per grid.
    if (p.publish && blockIdx.x == 0 && etid == 0) {
      if (generation_ok)
        p.state[1] = static_cast<int32_t>(g);
      else
        raise_flag(p.state, 0x4u);
    }
  }

  // --------------------------------------------------------------- teardown
  ptx::tc_fence_before();
  __syncthreads();
  if (S > 1) {
    // No CTA leaves while a peer may still address it: every thread arrived
    // after its last remote store, and this CTA's own receive barrier
    // completed, so the wait is normally immediate.
    __syncwarp();
    ptx::cluster_wait();
  }
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, p.tmem.cols);
  }
}

// programmatic: launched with programmatic stream serialisation, so the
// kernel may start (and stream W) before the previous kernel on the stream
// has finished.  Off where that kernel writes what the producer reads before
// its grid wait (the weight or its scale chunks).
template <int S, bool kWideLoad, int F, int T = 1>
cudaError_t launch_impl(const CUtensorMap& tmap_w, const CUtensorMap& tmap_x, const GemmParams& p,
                        cudaStream_t stream, bool programmatic) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((p.n / (kBlockN / F)) * S), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads_for_pipes(p.pipes)), 1, 1);
  cfg.dynamicSmemBytes = p.smem.total;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  int count = 0;
  if (programmatic) {
    attrs[count].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[count].val.programmaticStreamSerializationAllowed = 1;
    ++count;
  }
  if (S > 1) {
    attrs[count].id = cudaLaunchAttributeClusterDimension;
    attrs[count].val.clusterDim.x = S;
    attrs[count].val.clusterDim.y = 1;
    attrs[count].val.clusterDim.z = 1;
    ++count;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = count;
  return cudaLaunchKernelEx(&cfg, publish_gemm_kernel<S, kWideLoad, F, T>, tmap_w, tmap_x, p);
}

template <int S, bool kWideLoad, int F, int T = 1>
cudaError_t set_smem_impl(int bytes) {
  return cudaFuncSetAttribute(publish_gemm_kernel<S, kWideLoad, F, T>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

}  // namespace
}  // namespace mxfp8
