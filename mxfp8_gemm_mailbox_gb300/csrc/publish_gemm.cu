// Host side of the publishing GEMM: shared-memory and tensor-memory plans,
// the create-time re-layouts of W and its scales, and the launches of the
// unfolded kernels (the folded ones come from publish_gemm_fold.cu).
#include <algorithm>

#include "publish_gemm_kernel.cuh"

namespace mxfp8 {
namespace {

// W scales [n][k/32] -> [n/R][k_tiles][512] (R = 128 / fold rows per CTA,
// k_tiles = ceil(k / (128 fold))): inside a chunk, MMA row a and K block b of
// a 128-wide piece sit at byte (a % 32) * 16 + (a / 32) * 4 + b, the order the
// 32x128b tensor-memory copy and the MMA's scale lookup expect; MMA row a is
// weight row a % R of the tile in K piece a / R.  Blocks past K take 127.
__global__ void relayout_w_scales_kernel(const uint8_t* __restrict__ w_scale,
                                         uint8_t* __restrict__ w_sf, int n, int kblocks,
                                         int k_tiles, int fold) {
  const int rows = kBlockN / fold;
  const size_t total = static_cast<size_t>(n / rows) * k_tiles * kSfChunkBytes;
  for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t chunk = idx / kSfChunkBytes;
    const int within = static_cast<int>(idx % kSfChunkBytes);
    const int tile = static_cast<int>(chunk / k_tiles);
    const int kt = static_cast<int>(chunk % k_tiles);
    const int r0 = within / 16;
    const int r1 = (within % 16) / 4;
    const int b = within % 4;
    const int arow = r1 * 32 + r0;
    const int row = tile * rows + arow % rows;
    const int blk = (kt * fold + arow / rows) * kSfPerTile + b;
    w_sf[idx] = blk < kblocks ? w_scale[static_cast<size_t>(row) * kblocks + blk] : 127;
  }
}

// W [n][k] -> [n/R][k_tiles][16384]: each 16 KB block is the shared-memory
// image of one stage, 128 MMA rows x 128 bytes in the 128-byte swizzle (row a
// at byte a * 128, its 16-byte chunk c at position c ^ (a % 8)), MMA row a
// being weight row a % R of the tile in K piece a / R; one bulk copy lands it
// exactly as the fold's swizzled TMA boxes would.  Bytes past K are zero.
__global__ void tile_weights_kernel(const uint8_t* __restrict__ w, uint8_t* __restrict__ w_tiled,
                                    int n, int k, int k_tiles, int fold) {
  const int rows = kBlockN / fold;
  const size_t chunks = static_cast<size_t>(n / rows) * k_tiles * (kWTileBytes / 16);
  for (size_t q = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; q < chunks;
       q += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t block = q / (kWTileBytes / 16);
    const int within = static_cast<int>(q % (kWTileBytes / 16));
    const int tile = static_cast<int>(block / k_tiles);
    const int kt = static_cast<int>(block % k_tiles);
    const int a = within / 8;
    const int position = within % 8;
    const int c = position ^ (a & 7);
    const int k0 = (kt * fold + a / rows) * kTileK + c * 16;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (k0 < k)
      v = *reinterpret_cast<const uint4*>(w + static_cast<size_t>(tile * rows + a % rows) * k + k0);
    reinterpret_cast<uint4*>(w_tiled)[q] = v;
  }
}

}  // namespace

GemmSmemLayout gemm_smem_layout(int stages, int split_k, int tiles_per_split, int fold,
                                bool dedicated_recv, int tiles_per_stage) {
  GemmSmemLayout L{};
  const int ring_tiles = stages * tiles_per_stage;  // K tiles the rings hold
  L.w = 0;
  L.x = L.w + ring_tiles * kWTileBytes;
  L.sfa = L.x + ring_tiles * kXTileBytes * fold;
  // Written only after the main loop: the epilogue's BF16 tile in W stage 0,
  // the split-K partials from peers ((S-1) x 8/S x 128 x 8 bytes <= 6 KB) in
  // W stage 1 (every ring has at least two stages).
  L.ctile = L.w;
  L.recv = L.w + kWTileBytes;
  // One x scale chunk per stage (a 16-byte row per MMA column, two columns
  // to a row past 32 columns: 128 fold bytes, 512 at fold 8), plus the 384
  // bytes the copy of the last chunk reads past it (rows that feed no kept
  // column).
  L.sx = L.sfa + ring_tiles * kSfChunkBytes;
  const uint32_t sx_chunk = 16u * static_cast<uint32_t>(std::min(32, kRows * fold));
  const uint32_t sx_bytes = static_cast<uint32_t>(tiles_per_split) * sx_chunk + 384u;
  L.bars = (L.sx + sx_bytes + 7u) & ~7u;
  L.misc = L.bars + static_cast<uint32_t>(2 * stages + 2 * kMaxAccRing + 2) * 8u;
  L.total = L.misc + 16u + 1024u;
  if (dedicated_recv && split_k > 1) {
    // The partials' own region ((S-1) x 128 x 8/S pairs of 8 bytes, at most
    // 7 KB), so a peer can send them as soon as its own main loop is done.
    // 16-byte stores land there: keep it 16-byte aligned whatever precedes it.
    L.recv = (L.misc + 16u + 15u) & ~15u;
    L.recv_dedicated = 1;
    L.total = L.recv + static_cast<uint32_t>((split_k - 1) * kBlockN * (kRows / split_k) * 8) +
              1024u;
  }
  return L;
}

TmemPlan gemm_tmem_plan(int stages, int acc_blocks, int fold, int tiles_per_stage) {
  TmemPlan t{};
  t.acc = 0;
  const uint32_t block_cols = static_cast<uint32_t>(kRows * fold);  // one MMA's N
  t.acc_slot = acc_blocks == 1 ? kSfPerTile * block_cols : block_cols;
  // 32-column slots (fold 4) come 4 to a ring and 64-column ones (fold 8) 2,
  // so the plan stays within 256 columns.
  t.acc_ring = fold == 8 ? 2u
               : (acc_blocks == 1 || fold == 4) ? 4u
                                                : static_cast<uint32_t>(kMaxAccRing);
  // One 4-column W-scale and x-scale slot per K tile the ring holds.
  const uint32_t ring_tiles = static_cast<uint32_t>(stages * tiles_per_stage);
  t.sfa = t.acc + t.acc_slot * t.acc_ring;
  t.sfb = t.sfa + 4u * ring_tiles;
  const uint32_t used = t.sfb + 4u * ring_tiles;
  t.cols = 32;
  while (t.cols < used) t.cols <<= 1;
  return t;
}

cudaError_t set_gemm_smem_attribute(int split_k, int fold, int bytes, int tiles_per_stage) {
  if (tiles_per_stage == 2) return set_wide_stage_gemm_smem_attribute(split_k, fold, bytes);
  if (fold != 1) return set_folded_gemm_smem_attribute(split_k, fold, bytes);
  cudaError_t e = cudaSuccess;
  switch (split_k) {
    case 1:
      if ((e = set_smem_impl<1, false, 1>(bytes)) != cudaSuccess) return e;
      return set_smem_impl<1, true, 1>(bytes);
    case 2:
      if ((e = set_smem_impl<2, false, 1>(bytes)) != cudaSuccess) return e;
      return set_smem_impl<2, true, 1>(bytes);
    case 4:
      if ((e = set_smem_impl<4, false, 1>(bytes)) != cudaSuccess) return e;
      return set_smem_impl<4, true, 1>(bytes);
    case 8:
      if ((e = set_smem_impl<8, false, 1>(bytes)) != cudaSuccess) return e;
      return set_smem_impl<8, true, 1>(bytes);
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_publish_gemm(const CUtensorMap& tmap_w, const CUtensorMap& tmap_x,
                                const GemmParams& p, int split_k, cudaStream_t stream,
                                bool programmatic) {
  if (p.tiles_per_stage == 2)
    return launch_wide_stage_publish_gemm(tmap_w, tmap_x, p, split_k, stream, programmatic);
  if (p.fold != 1)
    return launch_folded_publish_gemm(tmap_w, tmap_x, p, split_k, stream, programmatic);
  const bool wide = p.tmem_load == MXFP8_TMEM_LOAD_16X256B;
  switch (split_k) {
    case 1:
      return wide ? launch_impl<1, true, 1>(tmap_w, tmap_x, p, stream, programmatic)
                  : launch_impl<1, false, 1>(tmap_w, tmap_x, p, stream, programmatic);
    case 2:
      return wide ? launch_impl<2, true, 1>(tmap_w, tmap_x, p, stream, programmatic)
                  : launch_impl<2, false, 1>(tmap_w, tmap_x, p, stream, programmatic);
    case 4:
      return wide ? launch_impl<4, true, 1>(tmap_w, tmap_x, p, stream, programmatic)
                  : launch_impl<4, false, 1>(tmap_w, tmap_x, p, stream, programmatic);
    case 8:
      return wide ? launch_impl<8, true, 1>(tmap_w, tmap_x, p, stream, programmatic)
                  : launch_impl<8, false, 1>(tmap_w, tmap_x, p, stream, programmatic);
    default:
      return cudaErrorInvalidValue;
  }
}

int k_tiles_for_fold(int k, int fold) {
  const int stage_k = kTileK * fold;
  return (k + stage_k - 1) / stage_k;
}

cudaError_t launch_tile_weights(const uint8_t* w, uint8_t* w_tiled, int n, int k, int fold,
                                cudaStream_t stream) {
  const int k_tiles = k_tiles_for_fold(k, fold);
  const size_t chunks =
      static_cast<size_t>(n / (kBlockN / fold)) * k_tiles * (kWTileBytes / 16);
  const int threads = 256;
  const int blocks = static_cast<int>(std::min<size_t>((chunks + threads - 1) / threads, 8192));
  tile_weights_kernel<<<blocks, threads, 0, stream>>>(w, w_tiled, n, k, k_tiles, fold);
  return cudaGetLastError();
}

cudaError_t launch_relayout_w_scales(const uint8_t* w_scale, uint8_t* w_sf, int n, int k,
                                     int fold, cudaStream_t stream) {
  const int k_tiles = k_tiles_for_fold(k, fold);
  const size_t total = static_cast<size_t>(n / (kBlockN / fold)) * k_tiles * kSfChunkBytes;
  const int threads = 256;
  const int blocks = static_cast<int>(std::min<size_t>((total + threads - 1) / threads, 4096));
  relayout_w_scales_kernel<<<blocks, threads, 0, stream>>>(w_scale, w_sf, n, k / 32, k_tiles,
                                                           fold);
  return cudaGetLastError();
}

}  // namespace mxfp8
