// Declarations shared by the kernels and the C-ABI layer of the library.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "mxfp8_mailbox.h"

namespace mxfp8 {

constexpr int kBlockN = 128;      // the MMA's M: output columns per CTA (128 / fold folded)
constexpr int kRows = 8;          // activation rows per x tile: the MMA's N (8 fold folded)
constexpr int kTileK = 128;       // K elements per stage piece: one 128-byte swizzle row
constexpr int kSfPerTile = 4;     // scale blocks of 32 per stage
// Warp 0 loads (one lane per pipe), warp 1 and warps 6.. issue MMAs (one
// warp per pipe), warps 2-5 run the epilogue.
constexpr int kMaxPipes = 4;
constexpr int kMaxThreads = 192 + 32 * (kMaxPipes - 1);
constexpr int threads_for_pipes(int pipes) { return 160 + 32 * pipes; }
constexpr int kSfChunkBytes = 512;
constexpr int kWTileBytes = kBlockN * kTileK;  // 16384
constexpr int kXTileBytes = kRows * kTileK;    // 1024
constexpr int kGenerations = 3;
constexpr uint32_t kSentinel = 0x80000000u;
constexpr int kMaxStages = 16;
constexpr int kMaxTilesPerSplit = 256;
constexpr int kMaxAccRing = 8;    // accumulator slots in tensor memory (one stage each)

// Byte offsets inside the GEMM's dynamic shared memory (after aligning the
// base to 1024 bytes), computed once on the host.
struct GemmSmemLayout {
  uint32_t w;         // stages x 16 KB W tiles
  uint32_t x;         // stages x 1 KB activation tiles
  uint32_t sfa;       // stages x 512 B W scale chunks
  uint32_t ctile;     // 8 x 128 BF16 epilogue staging (inside the dead W ring)
  uint32_t recv;      // split-K partials received from peers: in the dead W ring, or
                      // a region of its own when recv_dedicated
  uint32_t recv_dedicated;  // 1: peers may send before this CTA's main loop ends
  uint32_t sx;        // x scale chunks of this CTA's K range
  uint32_t bars;      // mbarriers
  uint32_t misc;      // tensor-memory base, generation broadcast
  uint32_t total;     // bytes including the alignment slack
};

// Tensor-memory columns of one CTA: the accumulator ring, then the W and x
// scale rings (4 columns a stage each).
struct TmemPlan {
  uint32_t cols;       // allocated (a power of two >= 32)
  uint32_t acc;        // first accumulator column
  uint32_t acc_slot;   // columns per accumulator slot (one stage of MMAs)
  uint32_t acc_ring;   // accumulator slots
  uint32_t sfa;        // first column of the W scale ring
  uint32_t sfb;        // first column of the x scale ring
};

struct GemmParams {
  int32_t n, k, m;
  int32_t k_tiles;          // K tiles: ceil(k / (128 fold))
  int32_t tiles_per_split;  // ceil(k_tiles / split_k)
  int32_t stages;
  int32_t capacity;
  int32_t publish;          // 1: fused publish into the mailbox; 0: C only
  int32_t acc_blocks;       // 32-wide K blocks summed in TMEM per promoted partial: 1 or 4
  int32_t l2_prefetch;      // stages past the ring warmed in L2 before the grid wait
  int32_t l2_prefetch_early;  // the same for CTAs with blockIdx.x < early_ctas
  int32_t early_ctas;       // the first CTAs, which launch beside the previous kernel
  int32_t pipes;            // producer lanes = MMA-issuing warps (1, 2, 4; divides stages)
  int32_t tmem_load;        // MXFP8_TMEM_LOAD_32X32B or MXFP8_TMEM_LOAD_16X256B
  int32_t fold;             // K pieces stacked in the MMA's 128 rows: 1, 2, 4 (128/fold
                            // output columns per CTA)
  int32_t x_pieces;         // 1: tmap_x is the 3-D piece view of x (a stage's F x
                            // tiles_per_stage pieces in one box); 0: the 2-D [m][k]
                            // view (one box per piece)
  int32_t tiles_per_stage;  // K tiles per pipeline stage: 1 (cta_k 128) or 2 (256)
  TmemPlan tmem;
  const uint8_t* x_scale;   // [m][k/32]
  const uint8_t* w_sf;      // [n/R][k_tiles][512] tiled W scales (R = 128 / fold)
  const uint8_t* w_tiled;   // [n/R][k_tiles][16384] shared-memory images of W, or nullptr
  uint16_t* c;              // [m][n] BF16 or nullptr
  const float* alpha;       // global scale of C (device scalar) or nullptr for 1
  uint16_t* mailbox;        // [3][capacity][n] BF16
  int32_t* state;           // int32[4]
  uint64_t wait_limit_ns;
  GemmSmemLayout smem;
};

// tiles_per_stage: 128-wide K tiles (of 128 fold K each) in one pipeline
// stage: 1 (cta_k 128) or 2 (cta_k 256).
GemmSmemLayout gemm_smem_layout(int stages, int split_k, int tiles_per_split, int fold,
                                bool dedicated_recv = false, int tiles_per_stage = 1);
TmemPlan gemm_tmem_plan(int stages, int acc_blocks, int fold, int tiles_per_stage = 1);
int k_tiles_for_fold(int k, int fold);  // ceil(k / (128 fold))

// Kernel launchers (return the CUDA error of the launch).  The GEMM's
// producer starts its weight and scale-chunk loads before the programmatic
// grid wait, so `programmatic` must be false when the kernel right before it
// on the stream may write those bytes.
cudaError_t launch_publish_gemm(const CUtensorMap& tmap_w, const CUtensorMap& tmap_x,
                                const GemmParams& p, int split_k, cudaStream_t stream,
                                bool programmatic);
cudaError_t set_gemm_smem_attribute(int split_k, int fold, int bytes, int tiles_per_stage);
cudaError_t launch_folded_publish_gemm(const CUtensorMap& tmap_w, const CUtensorMap& tmap_x,
                                       const GemmParams& p, int split_k, cudaStream_t stream,
                                       bool programmatic);
cudaError_t set_folded_gemm_smem_attribute(int split_k, int fold, int bytes);
// The cta_k 256 kernels (two K tiles per pipeline stage): fold 1, 2 or 4,
// split_k 1, 2 or 4, the 32x32b read-out.
cudaError_t launch_wide_stage_publish_gemm(const CUtensorMap& tmap_w, const CUtensorMap& tmap_x,
                                           const GemmParams& p, int split_k, cudaStream_t stream,
                                           bool programmatic);
cudaError_t set_wide_stage_gemm_smem_attribute(int split_k, int fold, int bytes);
cudaError_t launch_relayout_w_scales(const uint8_t* w_scale, uint8_t* w_sf, int n, int k,
                                     int fold, cudaStream_t stream);
cudaError_t launch_tile_weights(const uint8_t* w, uint8_t* w_tiled, int n, int k, int fold,
                                cudaStream_t stream);
cudaError_t launch_mailbox_init(uint16_t* mailbox, int32_t* state, int capacity, int n,
                                cudaStream_t stream);
cudaError_t launch_mailbox_consume(uint16_t* mailbox, int32_t* state, int capacity, int n, int m,
                                   uint16_t* out, uint64_t timeout_ns, cudaStream_t stream);
cudaError_t launch_lamport_gather_init(void* mailbox, int32_t* state, size_t capacity_bytes,
                                       cudaStream_t stream);
cudaError_t launch_lamport_gather(const void* in, void* out, void* mailbox, int32_t* state,
                                  size_t capacity_bytes, size_t nbytes, uint64_t timeout_ns,
                                  cudaStream_t stream);
cudaError_t launch_tagged_init(void* pairs, size_t bytes, cudaStream_t stream);
cudaError_t launch_tagged_publish(void* pairs, int n, int m, const uint16_t* c, uint32_t tag,
                                  cudaStream_t stream);
cudaError_t launch_tagged_consume(const void* pairs, int n, int m, uint32_t tag, uint16_t* out,
                                  uint64_t timeout_ns, int32_t* flags, cudaStream_t stream);
cudaError_t launch_mailbox_publish(uint16_t* mailbox, int32_t* state, int capacity, int n, int m,
                                   const uint16_t* c, cudaStream_t stream);

}  // namespace mxfp8
